// The whole MoE layer forward for decode batches (T <= kDecodeMaxT) in one
// persistent, cooperative launch of one CTA per SM.
//
// The kernel-chain forward launches route, dispatch, gather, two GEMMs and a
// combine; at one token the five non-GEMM launches cost about as much as the
// whole weight stream of a small layer.  Here the stages run as phases and
// tile tasks of one kernel, the single-kernel MoE layer idea of the CS349D
// lecture 8 notes (section 6, "FlashMoE：把分布式 MoE 层放进一个内核": one
// persistent kernel whose blocks take GEMM0 / GEMM1 / combine tile tasks,
// with no per-stage launches), on one GPU:
//
//   A  router      s = W_r x ("MoE推理优化全景指南", "从 Dense FFN 到专家集合"):
//                  CTA c computes the fp32 logits of experts c, c + G, ...
//                  for all T tokens (lane-strided products, a shuffle tree,
//                  the six warps' sums in order).
//      grid barrier
//   B  gating and dispatch, redundantly in every CTA (identical inputs and
//                  code, so identical results; no second barrier): top-k
//                  and gate weights per token (gating.cuh), then the counting
//                  dispatch ("MoE推理优化全景指南", "Dispatch 并不是一次普通
//                  all-to-all"): with T <= 16 each expert's tokens form a
//                  16-bit mask, count = popcount, offsets = prefix sum, and a
//                  token's position inside its expert's segment = popcount of
//                  the mask below it (ascending token order).  CTA 0 writes
//                  the routing metadata to the workspace.
//   C  expert GEMMs as tile tasks on the tensor cores (tcgen05, TMEM, TMA):
//                  gate/up tiles (128 gate + the same 128 up rows of one
//                  expert's W13, K = H) take x itself as the token operand --
//                  all T tokens, zero-filled to 16 rows, so no gather is
//                  needed -- and write h = SiLU(gate) * up for the expert's
//                  tokens; down tiles (256 rows of W2, K = I) take the
//                  expert's h rows and write the gate-weighted rows of
//                  out_perm.  The K steps of all tiles (gate/up first, then
//                  down) are cut into G equal contiguous ranges, one per CTA
//                  ("stream-K"), so every SM streams the same weight bytes;
//                  a tile shared by several CTAs is finished by the one
//                  holding its first K steps (it reaches the tile last),
//                  which adds the others' fp32 partials in CTA order.
//                  A down tile of expert e waits (bounded) until every
//                  gate/up tile of e has written its h rows; its weight
//                  copies are issued before that wait.
//      grid barrier
//   D  combine     y[t] = sum_j out_perm[inv_pos[t, j]] (+ the shared
//                  expert's row), fp32 in slot order, rounded once, spread
//                  over every thread of the grid.
//
// Every wait (grid barrier, expert readiness, pipeline barriers) gives up
// after kWaitLimitNs, latches kStatusTimeoutLayer in the status word and lets
// the CTA drain and exit; the cooperative launch guarantees that all CTAs are
// resident, which the cross-CTA waits rely on.
#include <string.h>

#include <cuda_fp8.h>

#include <mutex>

#include "gating.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kDThreads = 192;  // warps 0-3 epilogue, 4 TMA producer, 5 MMA
// FP8 weights: four more warps (6-9) convert the staged E4M3 weight tiles
// to the fp16 operand tiles the MMA reads
constexpr int kDThreads8 = 320;
constexpr int kDMaxWarps = kDThreads8 / 32;
constexpr uint32_t kDChunk = kBM * kBK * 2;                       // 128 rows x 64 bf16
constexpr uint32_t kDStageA = 2 * kStageKB * kDChunk;             // 64 KB of weights
constexpr uint32_t kDStageB = kStageKB * kDecodeMaxT * kBK * 2;   // 4 KB: 16 token rows
constexpr uint32_t kDStage = kDStageA + kDStageB;
constexpr int kDStages = 3;
constexpr uint32_t kDRing = kDStages * kDStage;
constexpr uint32_t kDTmemCols = 64;   // two buffers of two 16-column accumulators
constexpr int kDMaxAssign = kDecodeMaxT * kMaxK;
constexpr int kDSlotFloats = 2 * kBM * kDecodeMaxT;  // one split piece: 2 x 128 x 16 fp32
static_assert(kStageKB == 2, "a unit of work is two K blocks");
// FP8 ring: staging stages of one unit's E4M3 weights (two K blocks x 256
// rows x 64 bytes, 64-byte swizzled) filled by tensor copies, and operand
// stages of one K block.  An operand stage's weights (two 128-row halves x
// 64 fp16) are written by the converters into TMEM, where the MMA reads its
// A operand; only its 16 token rows (a tensor copy) are in shared memory.
constexpr uint32_t kF8Stage = 2 * 2 * kBM * kBK;           // 32 KB
constexpr int kF8Stages = 6;
constexpr uint32_t kOpStage = kDecodeMaxT * kBK * 2;       // 2 KB of token rows
constexpr int kOpStages = 4;
// TMEM of the FP8 layer: the accumulators in columns [0, 64), then per
// operand stage two halves of 32 columns (128 lanes = weight rows, a column
// = two fp16 of K)
constexpr uint32_t kF8ACol = 64;
constexpr uint32_t kF8AStageCols = 2 * kBK / 2;
constexpr uint32_t kDTmemColsF8 = 512;
static_assert(kF8ACol + kOpStages * kF8AStageCols <= kDTmemColsF8, "FP8 operands fit TMEM");
static_assert(kF8Stages * kF8Stage + kOpStages * kOpStage <= kDStages * kDStage,
              "the FP8 ring fits the stage ring");
static_assert((kF8Stages * kF8Stage) % 1024 == 0 && kOpStage % 1024 == 0,
              "staging and token tiles 1024-byte aligned");

struct DecodeMaps {
  CUtensorMap gu, gu_sh;  // W13 [E][2][I][H]: box 128 rows x 2 halves x 2 K blocks
  CUtensorMap dn, dn_sh;  // W2 [E][H][I]: box 256 rows x 2 K blocks
  CUtensorMap x;          // x [T][H]: box 16 rows x 2 K blocks (FP8 weights: 1)
  CUtensorMap h;          // h [R][I]: box 16 rows x 2 K blocks (FP8 weights: 1)
};

struct DecodeArgs {
  const __nv_bfloat16 *x;
  const float *w_router, *sel_bias;
  int T, H, E, k, I, gating, shared;
  float *logits, *topk_w, *gap, *w_perm;
  int32_t *ids, *counts, *offsets, *perm_src, *inv_pos;
  __nv_bfloat16 *h;
  __half *out_perm;
  __nv_bfloat16 *y;
  float *part;       // [2 * gridDim.x][kDSlotFloats] split-piece partials (per region)
  uint32_t *status;  // the workspace status block
  // FP8 weights: block exponents (scale 2^s per 128 x 128 block), W13
  // [E][2][ceil(I/128)][ceil(H/128)], W2 [E][ceil(H/128)][ceil(I/128)]
  const int8_t *s13, *s2, *s13_sh, *s2_sh;
  __half *x16;  // FP8 weights: x in fp16, the tensor-core operand of the gate/up tiles
};

// The two regions of work (all gate/up tiles, then all down tiles), each cut
// into Geff[r] equal contiguous ranges of granules, one per CTA: every CTA
// streams its share of the gate/up weights, then its share of the down
// weights.  A granule is one unit (a K step), or a whole tile where tiles
// have at most kDWholeTileUnits units: a tile split between CTAs costs a
// partial store, a release and the finishing CTA's wait, about as much as
// such a short tile itself (measured against unit granules: the TP-8 slice's
// down tiles, K = 192, at T=1 37.7 -> 35.4 us and T=4 63.5 -> 61.4 us; the
// tiny layer at T=16 32.1 -> 26.9 us; no change where tiles are longer).
constexpr int kDWholeTileUnits = 4;
struct Sched {
  int J[2], Uper[2], nt;  // tiles per segment, units per tile
  int U[2], Geff[2];      // units of the region (< 2^24), CTAs that share it
  int gran[2];            // units per granule
  int start[2], end[2];   // this CTA's unit range in each region
};

// Shared memory next to the stage ring.
struct DSmem {
  int32_t ids[kDMaxAssign];
  float w[kDMaxAssign];
  int32_t perm[kDMaxAssign];  // position -> assignment
  int32_t inv[kDMaxAssign];   // assignment -> position
  float wperm[kDMaxAssign];
  uint32_t mask[kMaxE];       // tokens of each expert (bit t)
  int32_t offs[kMaxE + 1];
  int32_t seg_list[kMaxE + 1];  // segments with rows, in order (shared expert last)
  float red[kDMaxWarps][kDecodeMaxT];
  int ntouched, last_flag, ok_flag;
  uint64_t full[kDStages], empty[kDStages], tfull[2], tempty[2], fin;
  uint64_t st_full[kF8Stages], st_empty[kF8Stages], op_full[kOpStages], op_empty[kOpStages];
  uint64_t rbar;  // router staging copies
  uint32_t tmem_slot;
  int abort_flag;
  Sched sc;  // indexed by region at run time: kept in shared memory
};
constexpr size_t kDSmemBytes = 1024 + kDRing + sizeof(DSmem);
static_assert(kDSmemBytes <= 232448, "shared memory per CTA");

// One contiguous range of units (pairs of K blocks) of one tile.
struct Piece {
  int dn;         // region: 0 gate/up tiles, 1 down tiles
  int seg, j;     // segment (expert; E = the shared expert) and row block
  int p0, p1;     // units [p0, p1) of the tile
  int tu;         // units of the tile
  int ts;         // first unit of the tile in its region
};

__device__ __forceinline__ Piece piece_at(const Sched &sc, const int32_t *seg_list, int r,
                                          int u) {
  Piece p;
  p.dn = r;
  const int q = u / sc.Uper[r];
  p.ts = q * sc.Uper[r];
  p.tu = sc.Uper[r];
  const int ti = q / sc.J[r];
  p.seg = seg_list[ti];
  p.j = q - ti * sc.J[r];
  p.p0 = u - p.ts;
  p.p1 = min(p.ts + p.tu, sc.end[r]) - p.ts;
  return p;
}

// Walks this CTA's pieces: region 0 (gate/up), then region 1 (down).
struct Cursor {
  int r, u;
};
__device__ __forceinline__ bool next_piece(const Sched &sc, const int32_t *seg_list, Cursor &c,
                                           Piece &p) {
  while (c.r < 2) {
    if (c.u < sc.end[c.r]) {
      p = piece_at(sc, seg_list, c.r, c.u);
      c.u = p.ts + p.p1;
      return true;
    }
    if (++c.r < 2) c.u = sc.start[c.r];
  }
  return false;
}

// The CTA whose range of region r holds unit x: with N = U / gran granules,
// the largest c with floor(c * N / Geff) <= x / gran.
__device__ __forceinline__ int cta_of(const Sched &sc, int r, int x) {
  const int64_t n = sc.U[r] / sc.gran[r], xg = x / sc.gran[r];
  return (int)(((xg + 1) * sc.Geff[r] + n - 1) / n - 1);
}

// Grid barrier over the CTAs of the (cooperative) launch, each of the two
// per launch on its own counter: every CTA adds 1 to it with a release
// reduction (no reply awaited) and polls it until it reaches `nblocks`; the
// last CTA to finish the kernel clears it.  Bounded: gives up after kWaitLimitNs, or at once when
// another CTA has latched a timeout, and then latches kStatusTimeoutLayer.
// Called by all threads.
__device__ bool grid_sync(uint32_t *bar, uint32_t nblocks, uint32_t *status, int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
      if (ld_acquire_gpu(bar) >= nblocks) break;
      if ((it & 15u) == 15u) {
        if (ld_acquire_gpu(status) & kStatusTimeoutMask) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(status, kStatusTimeoutLayer);
          ok = false;
          break;
        }
      }
    }
    *s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Bounded wait until a counter another CTA advances reaches `target`.
__device__ bool wait_counter(const uint32_t *cnt, uint32_t target, volatile int *abort_flag,
                             uint32_t *status) {
  if (ld_acquire_gpu(cnt) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_gpu(cnt) >= target) return true;
    if ((it & 15u) == 15u) {
      if (*abort_flag || (ld_acquire_gpu(status) & kStatusTimeoutMask)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeoutLayer);
        return false;
      }
    }
    __nanosleep(32);
  }
}

__device__ __forceinline__ void epi_sync_d() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool epi_all_d(bool p) {
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

// Two floats rounded to bf16 (round to nearest even), packed low first.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// y[t, col..col+8) = sum_j out_perm[inv[t*k + j], col..col+8) (+ the
// shared expert's row Na + t when nrow = k + 1), fp32 in slot order, rounded
// once to bf16; eight rows' loads in flight.
__device__ __forceinline__ void combine_vec(const DecodeArgs &a, const int32_t *inv, int k,
                                            int nrow, int Na, int H, int t, int col) {
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  for (int j0 = 0; j0 < nrow; j0 += 8) {
    uint4 raw[8];
#pragma unroll
    for (int z = 0; z < 8; ++z) {
      const int jj = j0 + z;
      if (jj < nrow) {
        const int pos = jj < k ? inv[t * k + jj] : Na + t;
        raw[z] = __ldcg(reinterpret_cast<const uint4 *>(a.out_perm + (size_t)pos * H + col));
      }
    }
#pragma unroll
    for (int z = 0; z < 8; ++z) {
      if (j0 + z < nrow) {
        const uint32_t wd[4] = {raw[z].x, raw[z].y, raw[z].z, raw[z].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&wd[q]));
          acc[2 * q] += f.x;
          acc[2 * q + 1] += f.y;
        }
      }
    }
  }
  uint4 o;
  o.x = bf16x2_bits(acc[0], acc[1]);
  o.y = bf16x2_bits(acc[2], acc[3]);
  o.z = bf16x2_bits(acc[4], acc[5]);
  o.w = bf16x2_bits(acc[6], acc[7]);
  *reinterpret_cast<uint4 *>(a.y + (size_t)t * H + col) = o;
}

// Four MMAs over one 64-deep K block (16 bf16 = 32 bytes per K16 step inside
// the 128-byte swizzled rows).
__device__ __forceinline__ void mma_kblock(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  umma_bf16(d, a, b, idesc, acc);
  umma_bf16(d, a + 2, b + 2, idesc, 1u);
  umma_bf16(d, a + 4, b + 4, idesc, 1u);
  umma_bf16(d, a + 6, b + 6, idesc, 1u);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, one CTA: A's rows in the TMEM lanes, two
// 16-bit elements of K per column.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One 64-deep K block with A in TMEM: four K16 steps of 8 columns.
__device__ __forceinline__ void mma_kblock_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                              uint32_t acc) {
  umma_ts(d, a, b, idesc, acc);
  umma_ts(d, a + 8, b + 2, idesc, 1u);
  umma_ts(d, a + 16, b + 4, idesc, 1u);
  umma_ts(d, a + 24, b + 6, idesc, 1u);
}

// 32 lanes x 32 consecutive 32-bit columns from registers; thread i writes
// lane (base + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
      " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Top-k and gate weights of every token into shared memory, one warp per
// token (NV logits per lane, E <= 32 * NV).
template <int NV>
__device__ __forceinline__ void gate_tokens(const DecodeArgs &a, int T, int E, int k,
                                            int32_t *ids, float *w, float *gap) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < T; t += (int)(blockDim.x >> 5)) {
    float s[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      s[i] = (e < E) ? __ldcg(a.logits + (size_t)t * E + e) : 0.f;
    }
    select_and_gate<NV>(s, lane, t, E, k, a.gating, a.sel_bias, ids, w, gap);
  }
}

// Two E4M3 codes (the low 16 bits of `two`) times 2^s as two fp16 values,
// packed low first: one conversion (E4M3 is a subset of fp16) and one fp16
// multiply by the power of two, exact for block exponents in [-15, 7].
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two, __half2 scale) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
  const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&hr), scale);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Instruction descriptor, kind::f16 with fp16 A and B (format 0 in bits 7-9
// and 10-12), fp32 accumulator (bits 4-5 = 1), both K-major, N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kDThreads8 : kDThreads, 1)
    decode_layer_kernel(const __grid_constant__ DecodeMaps maps, const DecodeArgs a) {
  constexpr int kNT = kFp8 ? kDThreads8 : kDThreads;  // threads of the CTA
  constexpr int kNW = kNT / 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  DSmem &S = *reinterpret_cast<DSmem *>(ring + kDRing);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.k, H = a.H, I = a.I;
  const int Na = T * k;
  const uint32_t G = gridDim.x;
  uint32_t *status = a.status;
  uint32_t *gbar = status + kDecodeBarrierWord;
  uint32_t *piece_cnt = status + kDecodePieceWord;
  uint32_t *seg_done = status + kDecodeSegWord;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.tfull[b], 1);
      mbar_init(&S.tempty[b], 4);
    }
    mbar_init(&S.fin, 1);
    mbar_init(&S.rbar, 1);
    if (kFp8) {
      for (int i = 0; i < kF8Stages; ++i) {
        mbar_init(&S.st_full[i], 1);   // the producer's expected bytes
        mbar_init(&S.st_empty[i], 4);  // the four converter warps
      }
      for (int i = 0; i < kOpStages; ++i) {
        mbar_init(&S.op_full[i], 5);   // token-row copy + four converter warps
        mbar_init(&S.op_empty[i], 1);  // the MMA's commit
      }
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&S.tmem_slot, kFp8 ? kDTmemColsF8 : kDTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&maps.gu);
    tma_prefetch_desc(&maps.gu_sh);
    tma_prefetch_desc(&maps.dn);
    tma_prefetch_desc(&maps.dn_sh);
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.h);
  }

  __syncthreads();  // barriers initialised before any thread waits on one

  // ---------------------------------------------------- A: router logits --
  // Work items are (expert e, group of tokens), at most about one per CTA:
  // the W_r row of e and the group's x rows are staged in shared memory (the
  // stage ring, idle until the GEMM phase) by bulk copies, in chunks of H
  // that fit, then every thread accumulates a strided part of H for every
  // token of the group; warp sums, then the six warps' sums in order.
  {
    const int per_e = max(1, (int)G / E);           // items per expert
    const int tpc = (T + per_e - 1) / per_e;        // tokens per item
    const int ngrp = (T + tpc - 1) / tpc;
    uint32_t rph = 0;
    for (int item = blockIdx.x; item < E * ngrp; item += G) {
      const int e = item / ngrp, t0 = (item - e * ngrp) * tpc;
      const int nt = min(tpc, T - t0);
      // H chunk: (nt rows of bf16 + one row of fp32) per column fits the ring
      int hc = (int)(kDRing / (uint32_t)(2 * nt + 4)) & ~63;
      if (hc > H) hc = H;
      float acc[kDecodeMaxT];
#pragma unroll
      for (int t = 0; t < kDecodeMaxT; ++t) acc[t] = 0.f;
      float *sw = reinterpret_cast<float *>(ring);
      uint16_t *sx = reinterpret_cast<uint16_t *>(ring + (size_t)hc * 4);
      for (int h0 = 0; h0 < H; h0 += hc) {
        const int hn = min(hc, H - h0);
        if (threadIdx.x == 0) {
          mbar_arrive_expect_tx(&S.rbar, (uint32_t)hn * (4 + 2 * nt));
          bulk_load(sw, a.w_router + (size_t)e * H + h0, (uint32_t)hn * 4, &S.rbar);
          for (int t = 0; t < nt; ++t)
            bulk_load(sx + (size_t)t * hc, a.x + (size_t)(t0 + t) * H + h0, (uint32_t)hn * 2,
                      &S.rbar);
        }
        if (!mbar_wait(&S.rbar, rph, &S.abort_flag, status, kStatusTimeoutLayer)) break;
        rph ^= 1u;
        for (int hh = threadIdx.x * 4; hh < hn; hh += kNT * 4) {
          const float4 wv = *reinterpret_cast<const float4 *>(sw + hh);
#pragma unroll
          for (int t = 0; t < kDecodeMaxT; ++t) {
            if (t < nt) {
              const uint2 raw = *reinterpret_cast<const uint2 *>(sx + (size_t)t * hc + hh);
              // bf16 -> fp32 is exact: the bf16 bits are the top half
              float v = acc[t];
              v = fmaf(wv.x, __uint_as_float(raw.x << 16), v);
              v = fmaf(wv.y, __uint_as_float(raw.x & 0xffff0000u), v);
              v = fmaf(wv.z, __uint_as_float(raw.y << 16), v);
              v = fmaf(wv.w, __uint_as_float(raw.y & 0xffff0000u), v);
              acc[t] = v;
            }
          }
        }
        // the chunk is consumed (generic reads ordered before the next bulk
        // copy's writes to the same shared memory) before the next copy lands
        fence_proxy_async_shared();
        __syncthreads();
      }
#pragma unroll
      for (int t = 0; t < kDecodeMaxT; ++t) {
        if (t < nt) {
          const float v = warp_sum(acc[t]);
          if (lane == 0) S.red[warp][t] = v;
        }
      }
      __syncthreads();
      if (warp == 0 && lane < nt) {
        float v = 0.f;
#pragma unroll
        for (int ww = 0; ww < kNW; ++ww) v += S.red[ww][lane];
        a.logits[(size_t)(t0 + lane) * E + e] = v;
      }
      __syncthreads();
    }
  }
  if (kFp8) {
    // x in fp16 for the gate/up tiles' tensor copies (exact for |x| in
    // [2^-14, 65504]; below, fp16's subnormal steps of 2^-24)
    const int64_t nv = (int64_t)T * H / 8;
    for (int64_t i = (int64_t)blockIdx.x * kNT + threadIdx.x; i < nv; i += (int64_t)G * kNT) {
      const uint4 r = reinterpret_cast<const uint4 *>(a.x)[i];
      const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __half2 hv = __floats2half2_rn(__uint_as_float(wd[q] << 16),
                                             __uint_as_float(wd[q] & 0xffff0000u));
        o[q] = *reinterpret_cast<const uint32_t *>(&hv);
      }
      reinterpret_cast<uint4 *>(a.x16)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_proxy_async_global();  // read by tensor copies after the barrier
  }
  bool ok = grid_sync(gbar, G, status, &S.ok_flag);
  if (kFp8) fence_proxy_async_global();

  // ------------------------------------------- B: gating and dispatch --
  if (ok) {
    const int nv = (E + 31) / 32;
    float *gap_out = blockIdx.x == 0 ? a.gap : nullptr;
    if (nv <= 1)
      gate_tokens<1>(a, T, E, k, S.ids, S.w, gap_out);
    else if (nv <= 2)
      gate_tokens<2>(a, T, E, k, S.ids, S.w, gap_out);
    else if (nv <= 4)
      gate_tokens<4>(a, T, E, k, S.ids, S.w, gap_out);
    else if (nv <= 8)
      gate_tokens<8>(a, T, E, k, S.ids, S.w, gap_out);
    else
      gate_tokens<16>(a, T, E, k, S.ids, S.w, gap_out);
    __syncthreads();
    if (warp == 0) {
      // the counting dispatch in one warp: per-expert token masks (the k
      // experts of a token are distinct), counts and offsets by a warp scan
      // over lane-owned expert ranges, then every assignment's position
      for (int e = lane; e < E; e += 32) S.mask[e] = 0u;
      __syncwarp();
      for (int i = lane; i < Na; i += 32) atomicOr(&S.mask[S.ids[i]], 1u << (i / k));
      __syncwarp();
      const int per = (E + 31) / 32;
      int sum = 0, nf = 0;
      for (int q = 0; q < per; ++q) {
        const int e = lane * per + q;
        if (e < E) {
          const int c = __popc(S.mask[e]);
          sum += c;
          nf += c > 0 ? 1 : 0;
        }
      }
      int incl = sum, inclf = nf;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        const int uf = __shfl_up_sync(0xffffffffu, inclf, o);
        if (lane >= o) {
          incl += u;
          inclf += uf;
        }
      }
      int run = incl - sum, frun = inclf - nf;
      for (int q = 0; q < per; ++q) {
        const int e = lane * per + q;
        if (e < E) {
          const int c = __popc(S.mask[e]);
          S.offs[e] = run;
          if (c > 0) S.seg_list[frun++] = e;
          run += c;
        }
      }
      if (lane == 31) {
        S.offs[E] = Na;
        int n = inclf;
        if (a.shared) S.seg_list[n++] = E;
        S.ntouched = n;
      }
      __syncwarp();
      for (int i = lane; i < Na; i += 32) {
        const int e = S.ids[i], t = i / k;
        const int pos = S.offs[e] + __popc(S.mask[e] & ((1u << t) - 1u));
        S.perm[pos] = i;
        S.inv[i] = pos;
        S.wperm[pos] = S.w[i];
      }
    }
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int i = threadIdx.x; i < Na; i += kNT) {
        a.ids[i] = S.ids[i];
        a.topk_w[i] = S.w[i];
        a.perm_src[i] = S.perm[i];
        a.inv_pos[i] = S.inv[i];
        a.w_perm[i] = S.wperm[i];
      }
      for (int e = threadIdx.x; e <= E; e += kNT) {
        a.offsets[e] = S.offs[e];
        if (e < E) a.counts[e] = __popc(S.mask[e]);
      }
    }
  }

  // ------------------------------------------------ C: expert GEMM tiles --
  if (threadIdx.x == 0) {
    Sched &w = S.sc;
    w.J[0] = (I + kBM - 1) / kBM;            // gate/up: 128 h columns per tile
    w.Uper[0] = (H / kBK + 1) / 2;           // K = H
    w.J[1] = (H + 2 * kBM - 1) / (2 * kBM);  // down: 256 W2 rows per tile
    w.Uper[1] = (I / kBK + 1) / 2;           // K = I
    w.nt = ok ? S.ntouched : 0;
    for (int r = 0; r < 2; ++r) {
      w.U[r] = w.nt * w.J[r] * w.Uper[r];
      w.gran[r] = w.Uper[r] <= kDWholeTileUnits ? w.Uper[r] : 1;
      const int n = w.U[r] / w.gran[r];  // granules of the region
      w.Geff[r] = min((int)G, n);
      if ((int)blockIdx.x < w.Geff[r]) {
        w.start[r] = (int)((int64_t)blockIdx.x * n / w.Geff[r]) * w.gran[r];
        w.end[r] = (int)(((int64_t)blockIdx.x + 1) * n / w.Geff[r]) * w.gran[r];
      } else {
        w.start[r] = w.end[r] = w.U[r];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_slot;
  const Sched &sc = S.sc;
  const int JG = sc.J[0];
  auto seg_row = [&](int s) { return s < E ? S.offs[s] : Na; };
  auto seg_rows = [&](int s) { return s < E ? S.offs[s + 1] - S.offs[s] : T; };

  if (kFp8 && warp == 4) {
    // ------------------------------------------- TMA producer, FP8 weights --
    // lane 0: each unit's E4M3 weights into the staging ring; lane 1: each
    // K block's token rows (x, or the expert's h rows once complete) into the
    // operand ring.  Two threads, so a down tile waiting for its h does not
    // hold back the weight copies behind it.
    if (lane == 0) {
      uint32_t st = 0, ph = 0, issued = 0;
      bool pok = true;
      Cursor cur = {0, sc.start[0]};
      Piece pc;
      while (pok && next_piece(sc, S.seg_list, cur, pc)) {
        const bool sh = pc.seg >= E;
        const CUtensorMap *ma =
            pc.dn ? (sh ? &maps.dn_sh : &maps.dn) : (sh ? &maps.gu_sh : &maps.gu);
        const int ecoord = sh ? 0 : pc.seg;
        const int arow = pc.dn ? pc.j * 2 * kBM : pc.j * kBM;
        for (int v = pc.p0; v < pc.p1; ++v) {
          if (!mbar_wait(&S.st_empty[st], ph ^ 1u, &S.abort_flag, status, kStatusTimeoutLayer)) {
            pok = false;
            break;
          }
          mbar_arrive_expect_tx(&S.st_full[st], kF8Stage);
          tma_load_5d(ring + st * kF8Stage, ma, &S.st_full[st], 0, arow, 0, 2 * v, ecoord);
          ++issued;
          if (++st == (uint32_t)kF8Stages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      const uint32_t n = issued < (uint32_t)kF8Stages ? issued : (uint32_t)kF8Stages;
      for (uint32_t i = 0; i < n; ++i) {
        st = st == 0 ? kF8Stages - 1 : st - 1;
        if (st == (uint32_t)kF8Stages - 1) ph ^= 1u;
        mbar_wait_drain(&S.st_full[st], ph);
      }
    } else if (lane == 1) {
      uint8_t *op = ring + kF8Stages * kF8Stage;
      uint32_t st = 0, ph = 0, issued = 0;
      bool pok = true;
      int ready = -1;  // last segment seen complete
      Cursor cur = {0, sc.start[0]};
      Piece pc;
      while (pok && next_piece(sc, S.seg_list, cur, pc)) {
        if (pc.dn && pc.seg != ready) {
          if (!wait_counter(seg_done + pc.seg, (uint32_t)JG, &S.abort_flag, status)) break;
          ready = pc.seg;
          fence_proxy_async_global();  // h was written by other CTAs' stores
        }
        const int row0 = seg_row(pc.seg);
        for (int v = pc.p0; pok && v < pc.p1; ++v) {
          for (int hk = 0; hk < kStageKB; ++hk) {
            if (!mbar_wait(&S.op_empty[st], ph ^ 1u, &S.abort_flag, status,
                           kStatusTimeoutLayer)) {
              pok = false;
              break;
            }
            mbar_arrive_expect_tx(&S.op_full[st], kOpStage);
            tma_load_3d(op + st * kOpStage, pc.dn ? &maps.h : &maps.x, &S.op_full[st], 0,
                        pc.dn ? row0 : 0, 2 * v + hk);
            ++issued;
            if (++st == (uint32_t)kOpStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      const uint32_t n = issued < (uint32_t)kOpStages ? issued : (uint32_t)kOpStages;
      for (uint32_t i = 0; i < n; ++i) {
        st = st == 0 ? kOpStages - 1 : st - 1;
        if (st == (uint32_t)kOpStages - 1) ph ^= 1u;
        mbar_wait_drain(&S.op_full[st], ph);
      }
    }
    __syncwarp();
  } else if (kFp8 && warp == 5) {
    // ----------------------------------------------- MMA issuer, FP8 weights --
    if (lane == 0) {
      uint8_t *op = ring + kF8Stages * kF8Stage;
      uint32_t st = 0, ph = 0, tl = 0;
      bool mok = true;
      const uint64_t desc0 = sdesc_k_sw128(smem_u32(op));
      const uint32_t id = idesc_f16_f32(kBM, kDecodeMaxT);  // fp16 x fp16 -> fp32
      Cursor cur = {0, sc.start[0]};
      Piece pc;
      for (; mok && next_piece(sc, S.seg_list, cur, pc); ++tl) {
        const uint32_t buf = tl & 1u, use = tl >> 1;
        if (!mbar_wait(&S.tempty[buf], (use & 1u) ^ 1u, &S.abort_flag, status,
                       kStatusTimeoutLayer))
          break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * 32u;
        for (int v = pc.p0; mok && v < pc.p1; ++v) {
          for (int hk = 0; hk < kStageKB; ++hk) {
            if (!mbar_wait(&S.op_full[st], ph, &S.abort_flag, status, kStatusTimeoutLayer)) {
              mok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bdesc = desc0 + st * (kOpStage >> 4);
            const uint32_t a0 = tmem_base + kF8ACol + st * kF8AStageCols;
            const uint32_t acc = (v != pc.p0 || hk != 0) ? 1u : 0u;
            // A from TMEM -- gate/up: gate rows, then up rows; down: W2 rows
            // [0,128), [128,256)
            mma_kblock_ts(d0, a0, bdesc, id, acc);
            mma_kblock_ts(d0 + 16, a0 + kF8AStageCols / 2, bdesc, id, acc);
            umma_commit(&S.op_empty[st]);
            if (++st == (uint32_t)kOpStages) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
        if (!mok) break;
        umma_commit(&S.tfull[buf]);
      }
      umma_commit(&S.fin);
      mbar_wait_drain(&S.fin, 0);
    }
    __syncwarp();
  } else if (kFp8 && warp >= 6) {
    // ------------------------------------------- converters (FP8 weights) --
    // Each K block of a staged unit: the two 128-row halves (128 rows x 64
    // E4M3 codes each) become 128 rows x 64 fp16, each code times its
    // block's scale, stored into the operand stage's TMEM columns, where the
    // MMA reads its A operand.  Warp w writes the TMEM lanes of its quarter
    // (w % 4), one weight row per thread: the row's 64 codes are four 16-byte
    // chunks, read through the 64-byte swizzle (so the warp's 32 rows touch
    // every bank once per phase), and become 32 columns of fp16 pairs.  The
    // MMA runs on fp16 operands: E4M3 codes convert to fp16 in one
    // instruction, and the token rows (x, h) are fp16 in this mode.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row of a 128-row half
    const int sw = (r >> 1) & 3;        // 64-byte swizzle of the staged rows
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16) + kF8ACol;
    uint32_t s1 = 0, p1 = 0, s2 = 0, p2 = 0;
    bool cok = true;
    const int nrb13 = (I + kBM - 1) / kBM, nkb13 = (H + kBM - 1) / kBM;
    const int nrb2 = (H + kBM - 1) / kBM, nkb2 = (I + kBM - 1) / kBM;
    Cursor cur = {0, sc.start[0]};
    Piece pc;
    while (cok && next_piece(sc, S.seg_list, cur, pc)) {
      const bool sh = pc.seg >= E;
      const int ex = sh ? 0 : pc.seg;
      for (int v = pc.p0; cok && v < pc.p1; ++v) {
        __half2 scl[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          int e8 = 0;
          if (!pc.dn) {
            e8 = (sh ? a.s13_sh : a.s13)[((ex * 2 + half) * nrb13 + pc.j) * nkb13 + v];
          } else if (2 * pc.j + half < nrb2) {  // (a half past H holds zero weights)
            e8 = (sh ? a.s2_sh : a.s2)[(ex * nrb2 + 2 * pc.j + half) * nkb2 + v];
          }
          scl[half] = __float2half2_rn(ldexpf(1.0f, e8));  // 2^e8, exact in fp16
        }
        if (!mbar_wait(&S.st_full[s1], p1, &S.abort_flag, status, kStatusTimeoutLayer)) {
          cok = false;
          break;
        }
        const uint8_t *src = ring + s1 * kF8Stage;
        for (int hk = 0; hk < kStageKB; ++hk) {
          if (!mbar_wait(&S.op_empty[s2], p2 ^ 1u, &S.abort_flag, status, kStatusTimeoutLayer)) {
            cok = false;
            break;
          }
          tc_fence_after();  // the MMAs that read this stage's columns are complete
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint8_t *rs = src + (hk * 2 + half) * (kBM * kBK) + r * kBK;
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 raw = *reinterpret_cast<const uint4 *>(rs + ((c ^ sw) << 4));
              const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                w[8 * c + 2 * q] = e4m3x2_to_f16x2(wd[q], scl[half]);
                w[8 * c + 2 * q + 1] = e4m3x2_to_f16x2(wd[q] >> 16, scl[half]);
              }
            }
            tmem_st32(lane_base + s2 * kF8AStageCols + half * (kF8AStageCols / 2), w);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.op_full[s2]);
          if (++s2 == (uint32_t)kOpStages) {
            s2 = 0;
            p2 ^= 1u;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.st_empty[s1]);
        if (++s1 == (uint32_t)kF8Stages) {
          s1 = 0;
          p1 ^= 1u;
        }
      }
    }
  } else if (warp == 4) {
    // ---------------------------------------------------- TMA producer --
    if (lane == 0) {
      uint32_t st = 0, ph = 0, issued = 0;
      bool pok = true;
      // token-row copies of down units queued until their expert's h is
      // complete (their weight copies are already in flight)
      int nq = 0;
      uint32_t q_st[kDStages];
      int q_seg[kDStages], q_row[kDStages], q_kb[kDStages];
      int ready = -1;  // last segment seen complete
      auto flush = [&]() -> bool {
        for (int i = 0; i < nq; ++i) {
          if (q_seg[i] != ready) {
            if (!wait_counter(seg_done + q_seg[i], (uint32_t)JG, &S.abort_flag, status))
              return false;
            ready = q_seg[i];
            fence_proxy_async_global();
          }
          tma_load_3d(ring + q_st[i] * kDStage + kDStageA, &maps.h, &S.full[q_st[i]], 0, q_row[i],
                      q_kb[i]);
        }
        nq = 0;
        return true;
      };
      Cursor cur = {0, sc.start[0]};
      Piece pc;
      while (pok && next_piece(sc, S.seg_list, cur, pc)) {
        const bool sh = pc.seg >= E;
        const CUtensorMap *ma =
            pc.dn ? (sh ? &maps.dn_sh : &maps.dn) : (sh ? &maps.gu_sh : &maps.gu);
        const int ecoord = sh ? 0 : pc.seg;
        const int arow = pc.dn ? pc.j * 2 * kBM : pc.j * kBM;
        const int row0 = seg_row(pc.seg);
        for (int v = pc.p0; v < pc.p1; ++v) {
          const int kb = 2 * v;
          if (nq > 0 && issued >= (uint32_t)kDStages && !flush()) {
            pok = false;
            break;
          }
          if (!mbar_wait(&S.empty[st], ph ^ 1u, &S.abort_flag, status, kStatusTimeoutLayer)) {
            pok = false;
            break;
          }
          uint8_t *dst = ring + st * kDStage;
          mbar_arrive_expect_tx(&S.full[st], kDStage);
          tma_load_5d(dst, ma, &S.full[st], 0, arow, 0, kb, ecoord);
          if (!pc.dn) {
            tma_load_3d(dst + kDStageA, &maps.x, &S.full[st], 0, 0, kb);
          } else {
            if (pc.seg != ready && nq == 0 &&
                ld_acquire_gpu(seg_done + pc.seg) >= (uint32_t)JG) {
              ready = pc.seg;
              fence_proxy_async_global();
            }
            if (pc.seg == ready && nq == 0) {
              tma_load_3d(dst + kDStageA, &maps.h, &S.full[st], 0, row0, kb);
            } else {
              q_st[nq] = st;
              q_seg[nq] = pc.seg;
              q_row[nq] = row0;
              q_kb[nq] = kb;
              ++nq;
            }
          }
          ++issued;
          if (++st == (uint32_t)kDStages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (pok && nq > 0) pok = flush();
      // drain: every issued copy lands before the CTA may exit
      const uint32_t n = issued < (uint32_t)kDStages ? issued : (uint32_t)kDStages;
      for (uint32_t i = 0; i < n; ++i) {
        st = st == 0 ? kDStages - 1 : st - 1;
        if (st == (uint32_t)kDStages - 1) ph ^= 1u;
        mbar_wait_drain(&S.full[st], ph);
      }
    }
    __syncwarp();
  } else if (!kFp8 && warp == 5) {
    // ------------------------------------------------------ MMA issuer --
    if (lane == 0) {
      uint32_t st = 0, ph = 0, tl = 0;
      bool mok = true;
      const uint64_t desc0 = sdesc_k_sw128(smem_u32(ring));
      const uint32_t id = idesc_bf16_f32(kBM, kDecodeMaxT);
      Cursor cur = {0, sc.start[0]};
      Piece pc;
      for (; mok && next_piece(sc, S.seg_list, cur, pc); ++tl) {
        const uint32_t buf = tl & 1u, use = tl >> 1;
        if (!mbar_wait(&S.tempty[buf], (use & 1u) ^ 1u, &S.abort_flag, status,
                       kStatusTimeoutLayer))
          break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * 32u;
        for (int v = pc.p0; v < pc.p1; ++v) {
          if (!mbar_wait(&S.full[st], ph, &S.abort_flag, status, kStatusTimeoutLayer)) {
            mok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = desc0 + st * (kDStage >> 4);
          const uint64_t bdesc = adesc + (kDStageA >> 4);
#pragma unroll
          for (int c = 0; c < kStageKB; ++c) {
            const uint32_t acc = (v != pc.p0 || c != 0) ? 1u : 0u;
            const uint64_t ac = adesc + c * ((2 * kDChunk) >> 4);
            const uint64_t bc = bdesc + c * ((kDecodeMaxT * kBK * 2) >> 4);
            // gate/up: gate rows, then up rows; down: W2 rows [0,128), [128,256)
            mma_kblock(d0, ac, bc, id, acc);
            mma_kblock(d0 + 16, ac + (kDChunk >> 4), bc, id, acc);
          }
          umma_commit(&S.empty[st]);
          if (++st == (uint32_t)kDStages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!mok) break;
        umma_commit(&S.tfull[buf]);
      }
      umma_commit(&S.fin);
      mbar_wait_drain(&S.fin, 0);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue --
    const int r = warp * 32 + lane;  // TMEM lane = weight row of the tile
    uint32_t tl = 0;
    bool range_bad = false;
    Cursor cur = {0, sc.start[0]};
    Piece pc;
    for (; next_piece(sc, S.seg_list, cur, pc); ++tl) {
      const uint32_t buf = tl & 1u, use = tl >> 1;
      const bool waited =
          mbar_wait(&S.tfull[buf], use & 1u, &S.abort_flag, status, kStatusTimeoutLayer);
      if (!epi_all_d(waited && !S.abort_flag)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + buf * 32u;
      uint32_t v0[16], v1[16];
      tmem_ld16(tb, v0);
      tmem_ld16(tb + 16, v1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tempty[buf]);  // the accumulator buffer is free
      float g[16], uu[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        g[q] = __uint_as_float(v0[q]);
        uu[q] = __uint_as_float(v1[q]);
      }
      const int s = pc.seg, row0 = seg_row(s), m = seg_rows(s);
      if (!(pc.p0 == 0 && pc.p1 == pc.tu)) {
        // A piece of a tile shared by CTAs c0..c1 (c0 holds the tile's first
        // units, at the end of its range: its piece comes last in time; the
        // others hold pieces at the start of theirs).  c1..c0+1 store the
        // fp32 partial of the live token columns (gate/up: the T tokens,
        // down: the segment's m rows) and signal with a release reduction;
        // c0 waits (bounded) for the c1 - c0 signals and adds the partials
        // to its own in CTA order.  No wait points to a piece that waits.
        const int ncol4 = ((pc.dn ? m : T) + 3) & ~3;
        const int c0 = cta_of(sc, pc.dn, pc.ts), c1 = cta_of(sc, pc.dn, pc.ts + pc.tu - 1);
        uint32_t *cnt = piece_cnt + pc.dn * kDecodeMaxCtas + c0;
        const size_t base = (size_t)pc.dn * kDSlotFloats + (size_t)r * 32;
        if ((int)blockIdx.x != c0) {
          float *mine = a.part + (size_t)(2 * blockIdx.x) * kDSlotFloats + base;
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            if (q < ncol4) {
              *reinterpret_cast<float4 *>(mine + q) =
                  make_float4(g[q], g[q + 1], g[q + 2], g[q + 3]);
              *reinterpret_cast<float4 *>(mine + 16 + q) =
                  make_float4(uu[q], uu[q + 1], uu[q + 2], uu[q + 3]);
            }
          }
          // release: the barrier orders every thread's partial before
          // thread 0's release reduction
          epi_sync_d();
          if (r == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
          continue;
        }
        // acquire: thread 0 sees all c1 - c0 signals, then the barrier
        // orders the reads below after its acquire
        if (r == 0) {
          const bool got = wait_counter(cnt, (uint32_t)(c1 - c0), &S.abort_flag, status);
          S.last_flag = got ? 1 : 0;
          if (got) *cnt = 0u;  // every signal of this launch has arrived
        }
        epi_sync_d();
        if (!S.last_flag) continue;
        // add the other pieces in CTA order; four slots' loads in flight
#pragma unroll
        for (int q = 0; q < 16; q += 4) {
          if (q < ncol4) {
            float4 ag = make_float4(g[q], g[q + 1], g[q + 2], g[q + 3]);
            float4 au = make_float4(uu[q], uu[q + 1], uu[q + 2], uu[q + 3]);
            for (int cc = c0 + 1; cc <= c1; cc += 4) {
              float4 lg[4], lu[4];
#pragma unroll
              for (int z = 0; z < 4; ++z) {
                lg[z] = lu[z] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (cc + z <= c1) {
                  const float *pp = a.part + (size_t)(2 * (cc + z)) * kDSlotFloats + base + q;
                  lg[z] = __ldcg(reinterpret_cast<const float4 *>(pp));
                  lu[z] = __ldcg(reinterpret_cast<const float4 *>(pp + 16));
                }
              }
#pragma unroll
              for (int z = 0; z < 4; ++z) {
                if (cc + z <= c1) {
                  ag.x += lg[z].x;
                  ag.y += lg[z].y;
                  ag.z += lg[z].z;
                  ag.w += lg[z].w;
                  au.x += lu[z].x;
                  au.y += lu[z].y;
                  au.z += lu[z].z;
                  au.w += lu[z].w;
                }
              }
            }
            g[q] = ag.x;
            g[q + 1] = ag.y;
            g[q + 2] = ag.z;
            g[q + 3] = ag.w;
            uu[q] = au.x;
            uu[q + 1] = au.y;
            uu[q + 2] = au.z;
            uu[q + 3] = au.w;
          }
        }
      }
      if (!pc.dn) {
        // h[row0 + n][j*128 + r] = SiLU(gate) * up of the segment's n-th token
        const int col = pc.j * kBM + r;
#pragma unroll
        for (int n = 0; n < kDecodeMaxT; ++n) {
          if (n < m) {
            const int t = s < E ? S.perm[row0 + n] / k : n;
            float gv = 0.f, uv = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              gv = (q == t) ? g[q] : gv;
              uv = (q == t) ? uu[q] : uv;
            }
            if (col < I) {
              const float hv = gv / (1.0f + __expf(-gv)) * uv;
              uint16_t bits;
              if (kFp8) {  // fp16 operand of the down tiles
                range_bad |= !(fabsf(hv) <= 65504.0f);
                bits = __half_as_ushort(__float2half_rn(fminf(fmaxf(hv, -65504.0f), 65504.0f)));
              } else {
                bits = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
              }
              reinterpret_cast<uint16_t *>(a.h)[(size_t)(row0 + n) * I + col] = bits;
            }
          }
        }
        // h is read by tensor copies (async proxy) of other CTAs' down tiles:
        // each writer orders its stores for the async proxy, the barrier
        // orders them before thread 0's release of the readiness count
        fence_proxy_async_global();
        epi_sync_d();
        if (r == 0)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(seg_done + s) : "memory");
      } else {
        // out_perm[row0 + n][j*256 + half*128 + r] = w_perm * (W2 h)
#pragma unroll
        for (int n = 0; n < kDecodeMaxT; ++n) {
          if (n < m) {
            const int pos = row0 + n;
            const float wv = pos < Na ? S.wperm[pos] : 1.0f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int col = pc.j * 2 * kBM + hh * kBM + r;
              const float val = (hh ? uu[n] : g[n]) * wv;
              range_bad |= !(fabsf(val) <= 65504.0f);
              if (col < H)
                a.out_perm[(size_t)pos * H + col] =
                    __float2half_rn(fminf(fmaxf(val, -65504.0f), 65504.0f));
            }
          }
        }
      }
    }
    if (range_bad) atomicOr(status, kStatusRange);
  }

  // ------------------------------------------------------- D: combine --
  // Once every CTA has written its down tiles' out_perm rows (a second grid
  // barrier), one vector of 8 columns per thread of the grid.  (Combining
  // each block of 256 columns in the CTA whose down tile completes it, with
  // no second barrier, left the combines of a batch on the few CTAs that
  // finish last.)
  if (ok) {
    ok = grid_sync(gbar + 1, G, status, &S.ok_flag);
    const int nvec = H / 8, nrow = k + a.shared;
    for (int task = (int)blockIdx.x * kNT + (int)threadIdx.x; ok && task < T * nvec;
         task += (int)G * kNT) {
      const int t = task / nvec;
      combine_vec(a, S.inv, k, nrow, Na, H, t, (task - t * nvec) * 8);
    }
  }

  // The last CTA to finish clears the grid barriers and the readiness
  // counters: every CTA has passed both barriers and its last readiness
  // check by then.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicInc(gbar + 2, G - 1) == G - 1) {  // wraps to 0
      __threadfence();
      gbar[0] = 0u;
      gbar[1] = 0u;
      for (int i = 0; i < sc.nt; ++i) seg_done[S.seg_list[i]] = 0u;
    }
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kFp8 ? kDTmemColsF8 : kDTmemCols);
  }
}

// Both CTAs of a two-CTA cooperative launch wait at a grid barrier sized for
// three: the waits run out and latch kStatusTimeoutLayer.
__global__ void __launch_bounds__(32) grid_wait_check_kernel(uint32_t *status) {
  __shared__ int s_ok;
  grid_sync(status + kDecodeBarrierWord, gridDim.x + 1, status, &s_ok);
  // (the barrier's count is left at gridDim.x: moe_workspace_init clears it)
}

// Tensor maps of one launch, cached by everything they depend on.
struct DecodeKey {
  int dev, T, H, E, I, k, shared, fp8;
  const void *w13, *w2, *w13s, *w2s, *x, *h;
  bool operator==(const DecodeKey &o) const { return memcmp(this, &o, sizeof o) == 0; }
};

bool decode_maps(const DecodeKey &key, DecodeMaps *out) {
  constexpr int kSlots = 8;
  static DecodeKey keys[kSlots];
  static DecodeMaps maps[kSlots];
  static bool used[kSlots] = {};
  static int next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < kSlots; ++i)
    if (used[i] && keys[i] == key) {
      *out = maps[i];
      return true;
    }
  DecodeMaps m;
  const int64_t R = (int64_t)key.T * key.k + (key.shared ? key.T : 0);
  auto wmap = key.fp8 ? weight_map_u8 : weight_map;
  if (!wmap(&m.gu, key.w13, key.H, key.I, 2, key.E, kBM)) return false;
  if (!wmap(&m.dn, key.w2, key.I, key.H, 1, key.E, 2 * kBM)) return false;
  if (key.shared) {
    if (!wmap(&m.gu_sh, key.w13s, key.H, key.I, 2, 1, kBM)) return false;
    if (!wmap(&m.dn_sh, key.w2s, key.I, key.H, 1, 1, 2 * kBM)) return false;
  } else {
    m.gu_sh = m.gu;
    m.dn_sh = m.dn;
  }
  // FP8 weights: operand stages of one K block
  const int kbl = key.fp8 ? 1 : kStageKB;
  if (!act_map(&m.x, key.x, key.H, key.T, kDecodeMaxT, kbl)) return false;
  if (!act_map(&m.h, key.h, key.I, R, kDecodeMaxT, kbl)) return false;
  keys[next] = key;
  maps[next] = m;
  used[next] = true;
  next = (next + 1) % kSlots;
  *out = m;
  return true;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_cooperative(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace

bool decode_layer_supported(const moe_layer_desc_t &d) {
  return d.T <= kDecodeMaxT && d.H >= 2 * kBM && (int64_t)d.T * d.k <= kDMaxAssign &&
         num_sms() <= kDecodeMaxCtas;
}

namespace {

// The weights of one launch, either format.
struct DecodeWeights {
  const float *w_router, *sel_bias;
  const void *w13, *w2, *w13s, *w2s;
  const int8_t *s13, *s2, *s13s, *s2s;  // FP8 only
};

template <bool kFp8>
cudaError_t launch_decode(const moe_layer_desc_t &d, const DecodeWeights &w,
                          const __nv_bfloat16 *x, __nv_bfloat16 *y, void *workspace,
                          const Layout &L, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeKey key;
  memset(&key, 0, sizeof key);
  key.dev = dev;
  key.T = d.T;
  key.H = d.H;
  key.E = d.E;
  key.I = d.I;
  key.k = d.k;
  key.shared = d.has_shared_expert ? 1 : 0;
  key.fp8 = kFp8 ? 1 : 0;
  key.w13 = w.w13;
  key.w2 = w.w2;
  key.w13s = key.shared ? w.w13s : nullptr;
  key.w2s = key.shared ? w.w2s : nullptr;
  // FP8 weights: the gate/up tiles read x in fp16, kept in the x_perm buffer
  // (which the persistent layer does not otherwise use)
  key.x = kFp8 ? static_cast<const void *>(ws + L.x_perm) : static_cast<const void *>(x);
  key.h = ws + L.h;
  DecodeMaps maps;
  if (!decode_maps(key, &maps)) return cudaErrorInvalidValue;
  DecodeArgs a;
  a.x = x;
  a.w_router = w.w_router;
  a.sel_bias = w.sel_bias;
  a.T = d.T;
  a.H = d.H;
  a.E = d.E;
  a.k = d.k;
  a.I = d.I;
  a.gating = d.gating;
  a.shared = key.shared;
  a.logits = reinterpret_cast<float *>(ws + L.logits);
  a.topk_w = reinterpret_cast<float *>(ws + L.topk_w);
  a.gap = reinterpret_cast<float *>(ws + L.gap);
  a.w_perm = reinterpret_cast<float *>(ws + L.w_perm);
  a.ids = reinterpret_cast<int32_t *>(ws + L.topk_ids);
  a.counts = reinterpret_cast<int32_t *>(ws + L.counts);
  a.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
  a.perm_src = reinterpret_cast<int32_t *>(ws + L.perm_src);
  a.inv_pos = reinterpret_cast<int32_t *>(ws + L.inv_pos);
  a.h = reinterpret_cast<__nv_bfloat16 *>(ws + L.h);
  a.out_perm = reinterpret_cast<__half *>(ws + L.out_perm);
  a.y = y;
  a.part = reinterpret_cast<float *>(ws + L.split_part);
  a.status = reinterpret_cast<uint32_t *>(ws + L.status);
  a.x16 = reinterpret_cast<__half *>(ws + L.x_perm);
  a.s13 = w.s13;
  a.s2 = w.s2;
  a.s13_sh = w.s13s;
  a.s2_sh = w.s2s;
  static bool configured[64] = {};
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel<kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kDSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_cooperative(decode_layer_kernel<kFp8>, dim3(num_sms()),
                            dim3(kFp8 ? kDThreads8 : kDThreads), kDSmemBytes, s, maps, a);
}

}  // namespace

cudaError_t launch_decode_layer(const moe_layer_desc_t &d, const moe_layer_weights_t &w,
                                const __nv_bfloat16 *x, __nv_bfloat16 *y, void *workspace,
                                const Layout &L, cudaStream_t s) {
  const DecodeWeights dw = {w.w_router, w.sel_bias, w.w13, w.w2, w.w13_shared, w.w2_shared,
                            nullptr,    nullptr,    nullptr, nullptr};
  return launch_decode<false>(d, dw, x, y, workspace, L, s);
}

cudaError_t launch_decode_layer_fp8(const moe_layer_desc_t &d, const moe_layer_weights_fp8_t &w,
                                    const __nv_bfloat16 *x, __nv_bfloat16 *y, void *workspace,
                                    const Layout &L, cudaStream_t s) {
  const DecodeWeights dw = {w.w_router,   w.sel_bias, w.w13,     w.w2,
                            w.w13_shared, w.w2_shared, w.w13_scale, w.w2_scale,
                            w.w13_shared_scale, w.w2_shared_scale};
  return launch_decode<true>(d, dw, x, y, workspace, L, s);
}

cudaError_t launch_grid_wait_check(uint32_t *status_block, cudaStream_t s) {
  return launch_cooperative(grid_wait_check_kernel, dim3(2), dim3(32), 0, s, status_block);
}

}  // namespace moe
