// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// The experts' SwiGLU FFNs run as two grouped GEMMs over the ragged
// per-expert row counts m_e ("MoE推理优化全景指南", section
// "Expert GEMM 为什么经常不够大": one scheduled launch computes
// [m_e, hidden] @ W_e for every expert; shapes W_gate/up[2I,H], W_down[H,I]
// from the Moebius reading notes, eq. (2)):
//
//   gate/up:  h[p, i]   = SiLU(sum_c W13[e][i][c] x[p][c]) * sum_c W13[e][I+i][c] x[p][c]
//   down:     out[p, r] = w_perm[p] * sum_i W2[e][r][i] h[p][i]
//
// Orientation ("swap AB"): the weight rows are the MMA's M = 128 dimension and
// the expert's token rows its N dimension.  In the decode regime an expert
// sees only a handful of rows, yet every weight byte is read from HBM once
// per (expert, 256-row token chunk) and streamed through the tensor cores at
// full M; in the prefill regime tiles are 128 x 256.
//
// Work unit (tile) = (segment s, weight-row block j, token chunk c); segments
// are the E experts (+ the shared expert, all T tokens).  A gate/up tile holds
// 64 gate rows and the 64 up rows of the same h columns (TMEM lanes [0, 64)
// and [64, 128)), so SiLU(gate)*up is formed in the epilogue and the two
// accumulators of a tile fit next to each other in TMEM; a down tile holds
// 128 rows of W2.  The tile plan (a prefix sum of tiles per segment, computed
// on the device from the dispatch offsets) is read by a persistent kernel,
// one CTA per SM, which walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// Tiles of one weight block are adjacent (chunk index innermost) so CTAs
// working at the same time share weight tiles through L2; experts with no
// rows have no tiles, so their weights are never read.
//
// CTA = 6 warps:
//   warp 4      TMA producer: a ring of pipeline stages (128-byte swizzle),
//               one per K step: the weight tile [128 x 64] and the tile's
//               token rows [16-row boxes, or whole 128-row halves, x 64];
//               completion on the stage's mbarrier.  Mostly-wide launches
//               (most token chunks over 128 rows) run 4 stages of 48 KB,
//               one per K step; others 6 stages of 32 KB, one per K step and
//               128-row half (decided on the device from the dispatch
//               counts);
//   warp 5      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma (bf16 in, fp32 accumulate in TMEM; one MMA per
//               128-token half and K16 step) and one tcgen05.commit per K
//               step, which frees the stage; the finished accumulator is
//               committed to the epilogue; two accumulator buffers of 256
//               columns let the epilogue of one tile overlap the mainloop of
//               the next;
//   warps 0-3   epilogue: tcgen05.ld of their 32 TMEM lanes, fused
//               SiLU(gate)*up (gate/up GEMM) or gate weighting (down GEMM),
//               bf16 (h) or fp16 (out_perm) stores.
// Every wait is bounded; on expiry the CTA records MOE_ERR_TIMEOUT's status
// bit, drains its copies and MMAs in flight, frees TMEM and returns.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {

// ---------------------------------------------------------- tensor maps --

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first,
// strides in bytes for dims 1..rank-1.
bool encode_bf16_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
              const cuuint64_t *strides, const cuuint32_t *box) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte tensor map (E4M3 codes) with 64-byte swizzle: in the 64-byte rows of
// a box, the 16-byte chunk c of row r lands at chunk c ^ ((r >> 1) & 3)
// (address bits 4-5 XOR bits 7-8), so a warp reading chunk c of 32
// consecutive rows, one row per thread, touches every bank once per phase.
static bool encode_u8_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                          const cuuint64_t *strides, const cuuint32_t *box) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void *>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


namespace {

constexpr int kThreads = 192;
constexpr uint32_t kChunkBytes = kBM * kBK * 2;  // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;              // two accumulators of 256 columns
constexpr uint32_t kAccCols = kTmemCols / 2;
// stage sizes (in units of kStageKB * 16 KB): gate/up 3, down 2 (narrow) or 3
// token rows of a thin stage (kStageKB K blocks x kThinRows rows)
constexpr uint32_t kThinB = kStageKB * kThinRows * kBK * 2;
// the most stages: thin down stages of 32 KB weights + kThinB
constexpr int kMaxStages = kRingBytes / (kStageKB * kChunkBytes + kThinB);
static_assert(kStageKB == 2, "stages are pairs of K blocks");
static_assert(kMaxStages == 5 && kRingBytes == 3 * (2 * kStageKB * kChunkBytes + kThinB),
              "ring: 3 thin gate/up stages, 5 thin down stages");
static_assert(kRingBytes >= 2 * 3 * kStageKB * kChunkBytes + 16 * 64 * 4 * 2,
              "wide gate/up: 2 stages of 96 KB and the up-value exchange buffer");

template <bool kGateUp>
struct Cfg {
  static constexpr uint32_t STAGE_UNIT = kStageKB * kChunkBytes;  // 128 rows of a stage
  static constexpr uint32_t SOUT_BYTES = 16 * kBM * 2;            // one 16-token slice (8 x kBM words)
  // gate/up, wide layout: up-row values handed to the gate rows' threads
  static constexpr uint32_t BAR_BYTES = (2 * kMaxStages + 5) * 8 + 16;
  static constexpr size_t smem_bytes(int nseg) {
    return 1024 + (size_t)kRingBytes + 2 * SOUT_BYTES + (size_t)kTileRowsDown * 4 +
           BAR_BYTES + (size_t)2 * (nseg + 1) * 4;
  }
  static_assert(smem_bytes(kMaxE + 1) <= 232448, "shared memory per CTA");
};

struct Tile {
  int seg, j, row0, nrows;
  bool wide;  // gate/up: 64 + 64 rows of W13 by up to 256 token rows
};

// Named barrier 1 over the 128 epilogue threads (warps 0-3).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The same barrier with an AND reduction: every epilogue thread gets the same
// answer, so all 128 take the same branch before the next epi_sync.
__device__ __forceinline__ bool epi_all(bool p) {
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

// Gate/up tiles are wide (64 + 64 rows of W13 by <= 256 token rows) in
// segments of more than `wide_above` rows, else 128 + 128 rows by <= 128
// token rows; down tiles are 128 rows of W2 by <= 256 token rows, or in the
// pair layout 256 rows by <= 128 (dn_rows = token rows per down tile).
template <bool kGateUp>
__device__ __forceinline__ Tile decode_tile(int tile, int wide_above, int dn_rows,
                                            const int32_t *seg_row, const int32_t *pref,
                                            int nseg) {
  int lo = 0, hi = nseg;  // pref[lo] <= tile < pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  Tile t;
  t.seg = lo;
  const int local = tile - pref[lo];
  const int m = seg_row[lo + 1] - seg_row[lo];
  t.wide = kGateUp && m > wide_above;
  const int rows = kGateUp ? (t.wide ? kTileRowsDown : kTileRowsGateUp) : dn_rows;
  const int chunks = (m + rows - 1) / rows;
  t.j = local / chunks;
  const int c = local - t.j * chunks;
  t.row0 = seg_row[lo] + c * rows;
  t.nrows = min(rows, m - c * rows);
  return t;
}

// Four MMAs: one 64-deep K block, 16 bf16 (32 bytes) per step inside the
// swizzled rows.
__device__ __forceinline__ void umma_kblock(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  umma_bf16(d, a, b, idesc, acc);
  umma_bf16(d, a + 2, b + 2, idesc, 1u);
  umma_bf16(d, a + 4, b + 4, idesc, 1u);
  umma_bf16(d, a + 6, b + 6, idesc, 1u);
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,     // routed weights (5D)
                       const __grid_constant__ CUtensorMap tm_a_sh,  // shared-expert weights (5D)
                       const __grid_constant__ CUtensorMap tm_aw,    // gate/up, wide: 64-row box
                       const __grid_constant__ CUtensorMap tm_aw_sh,
                       const __grid_constant__ TokenMaps tm_b,       // activations [R, K] (3D)
                       const int32_t *__restrict__ plan, int plan_early, int nseg, int E, int K,
                       int out_cols,
                       int64_t Na, const float *__restrict__ w_perm, void *__restrict__ out_,
                       float *__restrict__ split_part, uint32_t *__restrict__ split_cnt,
                       uint32_t *__restrict__ status) {
  using C = Cfg<kGateUp>;
  // gate/up writes h in bf16 (the next GEMM's operand); down writes the
  // gate-weighted rows in fp16: 11 significant bits (8x finer than bf16) at
  // the same bandwidth; magnitudes past the fp16 range are clamped and
  // latched in the status word.  Both are 2-byte elements.
  uint16_t *out = static_cast<uint16_t *>(out_);
  constexpr uint32_t kCode = kGateUp ? kStatusTimeoutGateUp : kStatusTimeoutDown;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *ring = smem;  // [stages][weights | token rows]
  uint16_t *sOut = reinterpret_cast<uint16_t *>(ring + kRingBytes);  // [2][8][kBM] words
  // wide gate/up: the up values handed to the gate rows' threads, [2][16][64],
  // in the ring's last 12 KB (two 96 KB stages leave them free)
  float *sUp = reinterpret_cast<float *>(ring + 2 * 3 * kStageKB * kChunkBytes);
  float *sW = reinterpret_cast<float *>(sOut + 2 * 16 * kBM);         // [kTileRowsDown] (down)
  uint64_t *full = reinterpret_cast<uint64_t *>(sW + kTileRowsDown);  // [kMaxStages]
  uint64_t *empty = full + kMaxStages;
  uint64_t *tfull = empty + kMaxStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *fin = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *s_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);  // last split piece
  int *s_kbs = reinterpret_cast<int *>(tmem_slot + 3);                     // K blocks per piece
  int32_t *seg_row = reinterpret_cast<int32_t *>(tmem_slot + 4);
  int32_t *pref = seg_row + nseg + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
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
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_sh);
    tma_prefetch_desc(&tm_aw);
    tma_prefetch_desc(&tm_aw_sh);
    for (int i = 0; i < 16; ++i) tma_prefetch_desc(&tm_b.m[i]);
  }
  // Everything above is independent of earlier kernels' outputs.  With
  // plan_early the tile plan was complete before the preceding kernel
  // started (it comes from an earlier kernel of the chain), so it is read
  // (through L2) before waiting on that kernel, and the producer requests its
  // first stages' weights before the wait too; only the token rows, the
  // preceding kernel's output, wait.
  const bool early = plan_early != 0;
  if (!early) {
    pdl_wait();
    pdl_launch_dependents();
  }
  const int32_t *g_pref = plan + (kGateUp ? 1 : 2) * (nseg + 1);
  for (int i = threadIdx.x; i <= nseg; i += blockDim.x) {
    seg_row[i] = __ldcg(plan + i);
    pref[i] = __ldcg(g_pref + i);
  }
  if (threadIdx.x == 0) *s_kbs = __ldcg(plan + 3 * (nseg + 1) + (kGateUp ? 0 : 1));
  // Stage layout of this launch (chosen by the tile plan).  Each stage holds
  // kStageKB K blocks of weights [K blocks][P][rows][64] and of token rows
  // [K blocks][rows][64]:
  //  - narrow: gate/up 128 gate + 128 up rows with <= 128 token rows; down
  //    128 rows with <= 128 token rows, a wider down tile then running one
  //    stage per 128-row half (its weights loaded once per half; the second
  //    load hits L2);
  //  - wide: gate/up 64 gate + 64 up rows, down 128 rows, with <= 256 token
  //    rows in one stage and one MMA per K16 step;
  //  - thin (every tile <= kThinRows token rows, the decode regime): narrow
  //    tiles with a token-row region of kThinRows rows, so 3 gate/up or 5
  //    down stages of weights are in flight instead of 2 or 3;
  //  - medium (down only, every tile <= kMediumRows token rows): 4 stages of
  //    128 rows + 64 token rows.
  const int layout = __ldcg(plan + 3 * (nseg + 1) + (kGateUp ? 2 : 3));
  const bool wide = layout == 1;
  // every tile <= kThinRows token rows (down: 5 = thin pair)
  const bool thin = layout == 2 || (!kGateUp && layout == 5);
  const bool medium = layout == 3;  // down: stages of 64 token rows
  // down, pair: 256 W2 rows (two 128-row halves) by <= 128 token rows
  const bool pair = !kGateUp && (layout == 4 || layout == 5);
  const int dn_rows = pair ? kBM : kTileRowsDown;  // token rows per down tile
  // token rows per stage: a down tile runs one stage per unit of this many
  // rows (gate/up tiles always fit one stage)
  const int unit_rows =
      kGateUp ? 256 : (wide ? 256 : (medium ? kMediumRows : (thin ? kThinRows : 128)));
  // gate/up: segments above this many rows get wide tiles (all of them in
  // the wide layout, the largest in the narrow one, none in the thin one)
  const int wide_above = wide ? 0 : (thin ? 1 << 30 : kGateUpWideAbove);
  // gate/up stages: 96 KB for either tile shape (64 KB weights + 32 KB token
  // rows, or 32 + 64 KB), thin 64 + 4 KB; down stages: 32 KB weights + the
  // layout's token rows
  const uint32_t U = C::STAGE_UNIT;
  const uint32_t stage_bytes =
      kGateUp ? (thin ? 2 * U + kThinB : 3 * U)
              : (pair ? (thin ? 2 * U + kThinB : 3 * U)
                      : U + (thin ? kThinB : medium ? U / 2 : (wide ? 2 : 1) * U));
  const uint32_t nst = kRingBytes / stage_bytes;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (early && warp != 4) {
    pdl_wait();
    pdl_launch_dependents();
  }
  const uint32_t tmem_base = *tmem_slot;
  // the stage ring must hold one to kMaxStages stages of this layout (the
  // barrier arrays have kMaxStages entries); otherwise report and stop
  if (nst < 1 || nst > (uint32_t)kMaxStages) {
    if (threadIdx.x == 0) atomicOr(status, kCode);
    if (warp == 5) tmem_dealloc(tmem_base, kTmemCols);
    return;
  }
  const int total = pref[nseg];
  const int nkb = K / kBK;
  // work unit = one K piece of a tile: kbs K blocks (the whole tile, or an
  // even number when the plan splits K)
  const int kbs = *s_kbs;
  const int S = (nkb + kbs - 1) / kbs;
  const int total_pieces = total * S;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer --
    // Per stage: the weight rows of the tile in one copy and its token rows
    // [K blocks][h][64] in one copy, h = rows rounded up to 16 (a 128-row
    // half of a wider down tile in the narrow layout).
    if (lane == 0) {
      uint32_t st = 0, ph = 0, issued = 0;  // stage, parity of its use, stages issued
      bool ok = true;
      // before the wait on the preceding kernel (plan_early): the first nst
      // stages' token-row copies are queued and issued after it
      bool waiting = early;
      int nq = 0;
      uint32_t q_st[kMaxStages];
      int q_row[kMaxStages], q_h[kMaxStages], q_kb[kMaxStages], q_off[kMaxStages];
      auto release_queue = [&]() {
        pdl_wait();
        pdl_launch_dependents();
        for (int i = 0; i < nq; ++i)
          tma_load_3d(ring + q_st[i] * stage_bytes + q_off[i], &tm_b.m[(q_h[i] >> 4) - 1],
                      &full[q_st[i]], 0, q_row[i], q_kb[i]);
        nq = 0;
        waiting = false;
      };
      for (int pc = blockIdx.x; ok && pc < total_pieces; pc += gridDim.x) {
        const int tile = pc / S, z = pc - tile * S;
        const Tile t = decode_tile<kGateUp>(tile, wide_above, dn_rows, seg_row, pref, nseg);
        const int kb0 = z * kbs, kb1 = min(nkb, kb0 + kbs);
        const bool sh = (t.seg >= E);
        // gate/up wide tiles and down pair tiles take the second pair of maps
        // (64-row and 256-row boxes)
        const CUtensorMap *ma =
            (t.wide || pair) ? (sh ? &tm_aw_sh : &tm_aw) : (sh ? &tm_a_sh : &tm_a);
        const int ecoord = sh ? 0 : t.seg;
        // this tile's weight bytes per stage (and offset of its token rows)
        const bool two = (kGateUp && !t.wide) || pair;  // two 128-row A halves
        const uint32_t stage_a = two ? 2 * U : U;
        const int arow = t.j * (t.wide ? kGateUpColsWide : (pair ? 2 * kBM : kBM));
        const int n16 = (t.nrows + 15) & ~15;       // token rows, padded to 16
        const int nu = (n16 + unit_rows - 1) / unit_rows;  // stages per K step
        for (int kb = kb0; ok && kb < kb1; kb += kStageKB) {
          for (int u = 0; u < nu; ++u) {
            if (waiting && issued == nst) release_queue();  // before any stage is reused
            if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, status, kCode)) {
              ok = false;
              break;
            }
            uint8_t *dst = ring + st * stage_bytes;
            // token rows of this stage: unit u of the tile
            const int hb = min(unit_rows, n16 - u * unit_rows);
            mbar_arrive_expect_tx(&full[st], stage_a + (uint32_t)hb * (kStageKB * kBK * 2));
            // [K blocks][P][rows][64]: gate/up P = 2 (gate rows, then the same
            // up rows), down P = 1
            tma_load_5d(dst, ma, &full[st], 0, arow, 0, kb, ecoord);
            if (waiting) {
              q_st[nq] = st;
              q_row[nq] = t.row0 + u * unit_rows;
              q_h[nq] = hb;
              q_kb[nq] = kb;
              q_off[nq] = (int)stage_a;
              ++nq;
            } else {
              tma_load_3d(dst + stage_a, &tm_b.m[(hb >> 4) - 1], &full[st], 0,
                          t.row0 + u * unit_rows, kb);
            }
            ++issued;
            if (++st == nst) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (waiting) release_queue();
      // Drain: every issued copy must land before the CTA may exit.
      const uint32_t n = issued < nst ? issued : nst;
      for (uint32_t i = 0; i < n; ++i) {
        // the n most recent uses, newest first
        st = st == 0 ? nst - 1 : st - 1;
        if (st == nst - 1) ph ^= 1u;
        mbar_wait_drain(&full[st], ph);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t st = 0, ph = 0, tl = 0;  // stage, parity, tiles
      // stage descriptors differ only in the start-address field (16-byte units)
      const uint64_t desc0 = sdesc_k_sw128(smem_u32(ring));
      const uint32_t dstage = stage_bytes >> 4;
      bool ok = true;
      for (int pc = blockIdx.x; ok && pc < total_pieces; pc += gridDim.x, ++tl) {
        const int tile = pc / S, z = pc - tile * S;
        const Tile t = decode_tile<kGateUp>(tile, wide_above, dn_rows, seg_row, pref, nseg);
        const int kb0 = z * kbs, kb1 = min(nkb, kb0 + kbs);
        const int n16 = (t.nrows + 15) & ~15;
        const int nu = (n16 + unit_rows - 1) / unit_rows;
        const bool two = (kGateUp && !t.wide) || pair;  // two 128-row A halves
        const uint32_t stage_a = two ? 2 * U : U;          // this tile's weights
        const uint32_t chunk_a = stage_a / kStageKB;                   // per K block
        // token column n -> accumulator column n (a wide down tile in the
        // narrow layout as two 128-row units); gate/up, narrow: gate rows ->
        // columns [0, 128), up rows -> [128, 256) of the same token; gate/up,
        // wide: one accumulator, gate rows in lanes [0, 64), up in [64, 128)

        const uint32_t buf = tl & 1u, use = tl >> 1;
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, status, kCode)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * kAccCols;
        for (int kb = kb0; ok && kb < kb1; kb += kStageKB) {
          const int nc = min(kStageKB, kb1 - kb);  // K blocks of this piece in the stage
          for (int u = 0; u < nu; ++u) {
            if (!mbar_wait(&full[st], ph, abort_flag, status, kCode)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t adesc = desc0 + st * dstage;
            const uint64_t bdesc = adesc + (stage_a >> 4);
            const int hb = min(unit_rows, n16 - u * unit_rows);
            const uint32_t id = idesc_bf16_f32(kBM, hb);
            for (int c = 0; c < nc; ++c) {
              const uint32_t acc = (kb != kb0 || c != 0) ? 1u : 0u;
              const uint64_t ac = adesc + c * (chunk_a >> 4);
              const uint64_t bc = bdesc + c * ((uint32_t)hb * (kBK * 2) >> 4);
              if (two) {
                // gate/up: gate rows, up rows; down pair: W2 rows [0,128), [128,256)
                umma_kblock(d0, ac, bc, id, acc);
                umma_kblock(d0 + 128, ac + (kChunkBytes >> 4), bc, id, acc);
              } else {
                // one MMA over all of the stage's token rows (N <= 256)
                umma_kblock(d0 + (uint32_t)(u * unit_rows), ac, bc, id, acc);
              }
            }
            umma_commit(&empty[st]);  // the stage is free once these MMAs have read it
            if (++st == nst) {
              st = 0;
              ph ^= 1u;
            }
          }
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);  // accumulator complete
      }
      umma_commit(fin);  // every MMA issued above has completed
      mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    // Per 16-token slice: tcgen05.ld of the thread's accumulator row(s) (16
    // token columns), fused SiLU(gate)*up or gate weighting, the slice
    // written transposed into smem (two buffers, alternating), then stored
    // as token rows with 16-byte vector stores by all 128 epilogue threads.
    // A split-K piece instead writes its fp32 partial; the last piece of the
    // tile adds the S partials in split order and runs the same epilogue.
    const int r = warp * 32 + lane;  // TMEM lane = weight row of the tile
    uint32_t tl = 0, slice = 0;
    // down: the largest magnitude written (NaN-propagating), checked once
    float vmax = 0.f;
    // A 16-token slice goes through smem as 32-bit words [8 token pairs][kBM
    // columns]: word (p, r) holds column r of tokens n0 + 2p (low half) and
    // n0 + 2p + 1 (high half), so each thread converts two values per
    // instruction and stores one word per token pair.  Then every thread
    // takes one (token pair, 8-column chunk), splits the halves apart with
    // byte permutes and stores 16 bytes to each token's row.
    auto emit16 = [&](const Tile &t, int n0, int col0, const float(&g)[16],
                      const float(&u)[16]) {
      uint32_t *so = reinterpret_cast<uint32_t *>(sOut) + (slice & 1u) * (8 * kBM);
      float wv[16];
      if (!kGateUp) {
#pragma unroll
        for (int q = 0; q < 16; q += 4) {
          const float4 a = *reinterpret_cast<const float4 *>(sW + n0 + q);
          wv[q] = a.x;
          wv[q + 1] = a.y;
          wv[q + 2] = a.z;
          wv[q + 3] = a.w;
        }
      }
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        uint32_t word;
        if (kGateUp) {
          const float g0 = g[2 * p], g1 = g[2 * p + 1];
          word = pack_bf16x2(__fdividef(g0, 1.0f + __expf(-g0)) * u[2 * p],
                             __fdividef(g1, 1.0f + __expf(-g1)) * u[2 * p + 1]);
        } else {
          const float v0 = g[2 * p] * wv[2 * p], v1 = g[2 * p + 1] * wv[2 * p + 1];
          // every column counts: the token rows a tile reads past its own
          // are another segment's, zero-filled past the tensor, or zeroed by
          // the gather past the last segment (measured: checking only the
          // stored columns made the TP-8 slice's down GEMM 3-70% slower)
          vmax = fmax_nan(vmax, fabsf(v0));
          vmax = fmax_nan(vmax, fabsf(v1));
          // magnitudes past the fp16 range saturate to +-65504
          word = pack_f16x2_satfinite(v0, v1);
        }
        so[p * kBM + r] = word;
      }
      epi_sync();
      const int p = r >> 4, ch = r & 15;  // 8 token pairs x 16 chunks of 8 columns
      const uint4 lo = *reinterpret_cast<const uint4 *>(so + p * kBM + ch * 8);
      const uint4 hi = *reinterpret_cast<const uint4 *>(so + p * kBM + ch * 8 + 4);
      const uint4 a = make_uint4(__byte_perm(lo.x, lo.y, 0x5410), __byte_perm(lo.z, lo.w, 0x5410),
                                 __byte_perm(hi.x, hi.y, 0x5410), __byte_perm(hi.z, hi.w, 0x5410));
      const uint4 b = make_uint4(__byte_perm(lo.x, lo.y, 0x7632), __byte_perm(lo.z, lo.w, 0x7632),
                                 __byte_perm(hi.x, hi.y, 0x7632), __byte_perm(hi.z, hi.w, 0x7632));
      const int n = n0 + 2 * p, col = col0 + ch * 8;
      if (col < out_cols) {
        uint16_t *o = out + ((int64_t)t.row0 + n) * out_cols + col;
        if (n < t.nrows) *reinterpret_cast<uint4 *>(o) = a;
        if (n + 1 < t.nrows) *reinterpret_cast<uint4 *>(o + out_cols) = b;
      }
      ++slice;
    };
    // gate/up, wide layout: the thread holds a gate row (r < 64) or the up row
    // r - 64 of the same h column; the up values pass through smem.
    auto emit16_wide = [&](const Tile &t, int n0, const float(&v)[16]) {
      constexpr int W = kGateUpColsWide;
      uint16_t *so = sOut + (slice & 1u) * (16 * kBM);  // [16][W]
      float *su = sUp + (slice & 1u) * (16 * W);
      if (r >= W) {
#pragma unroll
        for (int q = 0; q < 16; ++q) su[q * W + (r - W)] = v[q];
      }
      epi_sync();
      if (r < W) {
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float g = v[q], u = su[q * W + r];
          so[q * W + r] = __bfloat16_as_ushort(__float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u));
        }
      }
      epi_sync();
      // 16 token rows x 64 columns x 2 bytes = 128 chunks of 16 bytes
      const int q = r / (W / 8), ch = r % (W / 8);
      const int n = n0 + q, col = t.j * W + ch * 8;
      if (n < t.nrows && col < out_cols)
        *reinterpret_cast<uint4 *>(out + ((int64_t)t.row0 + n) * out_cols + col) =
            *reinterpret_cast<const uint4 *>(so + q * W + ch * 8);
      ++slice;
    };
    // floats of one split-K piece's partial (a split launch is never wide:
    // the plan splits only when every tile has <= kSplitMaxRows rows); two
    // accumulators for gate/up and for the down pair layouts
    const bool two_acc = kGateUp || pair;
    const int slot = (two_acc ? 2 : 1) * kBM * kSplitMaxRows;
    for (int pc = blockIdx.x; pc < total_pieces; pc += gridDim.x, ++tl) {
      const int tile = pc / S, z = pc - tile * S;
      const Tile t = decode_tile<kGateUp>(tile, wide_above, dn_rows, seg_row, pref, nseg);
      const uint32_t buf = tl & 1u, use = tl >> 1;
      const bool waited = mbar_wait(&tfull[buf], use & 1u, abort_flag, status, kCode);
      // one decision for all 128 epilogue threads: they share named barriers
      if (!epi_all(waited && !*abort_flag)) break;
      tc_fence_after();
      if (!kGateUp) {
        for (int n = r; n < kTileRowsDown; n += 128) {
          const int64_t row = (int64_t)t.row0 + n;
          // routed segments: the gate weight; the shared expert: weight 1
          sW[n] = (n < t.nrows && w_perm != nullptr && t.seg < E && row < Na) ? w_perm[row]
                                                                              : 1.0f;
        }
        epi_sync();
      }
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + buf * kAccCols;
      const int N = (t.nrows + 15) & ~15;
      if (kGateUp && t.wide) {
        for (int n0 = 0; n0 < N; n0 += 16) {
          uint32_t v0[16];
          tmem_ld16(tb + n0, v0);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = __uint_as_float(v0[q]);
          emit16_wide(t, n0, v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        continue;
      }
      if (S == 1) {
        // down pair: the second 128-row half's columns follow at +128
        for (int h = 0; h < (pair ? 2 : 1); ++h) {
          const int col0 = pair ? t.j * 2 * kBM + h * kBM : t.j * kBM;
          for (int n0 = 0; n0 < N; n0 += 16) {
            uint32_t v0[16], v1[16];
            tmem_ld16(tb + h * 128 + n0, v0);
            if (kGateUp) tmem_ld16(tb + 128 + n0, v1);
            tmem_ld_wait();
            float g[16], u[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              g[q] = __uint_as_float(v0[q]);
              u[q] = kGateUp ? __uint_as_float(v1[q]) : 0.f;
            }
            emit16(t, n0, col0, g, u);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        continue;
      }
      // ---- split-K piece (N <= kSplitMaxRows): fp32 partial to global ----
      float *part = split_part + (size_t)(tile * S + z) * slot + (size_t)r * kSplitMaxRows;
      for (int n0 = 0; n0 < N; n0 += 16) {
        uint32_t v0[16], v1[16];
        tmem_ld16(tb + n0, v0);
        if (two_acc) tmem_ld16(tb + 128 + n0, v1);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; q += 4) {
          *reinterpret_cast<float4 *>(part + n0 + q) =
              make_float4(__uint_as_float(v0[q]), __uint_as_float(v0[q + 1]),
                          __uint_as_float(v0[q + 2]), __uint_as_float(v0[q + 3]));
          if (two_acc)
            *reinterpret_cast<float4 *>(part + kBM * kSplitMaxRows + n0 + q) =
                make_float4(__uint_as_float(v1[q]), __uint_as_float(v1[q + 1]),
                            __uint_as_float(v1[q + 2]), __uint_as_float(v1[q + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      epi_sync();  // every partial store of this CTA precedes the fence below
      // release the partial, arrive; atomicInc wraps to 0 at the last piece,
      // so the counter is ready for the next call
      if (r == 0) {
        __threadfence();
        *s_flag = (atomicInc(&split_cnt[tile], S - 1) == (unsigned)(S - 1));
      }
      epi_sync();
      if (!*s_flag) continue;
      __threadfence();
      for (int n0 = 0; n0 < N; n0 += 16) {
        float g[16], u[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) g[q] = u[q] = 0.f;
        for (int zz = 0; zz < S; ++zz) {
          const float *p =
              split_part + (size_t)(tile * S + zz) * slot + (size_t)r * kSplitMaxRows + n0;
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(p + q));
            g[q] += a.x;
            g[q + 1] += a.y;
            g[q + 2] += a.z;
            g[q + 3] += a.w;
            if (two_acc) {
              const float4 b = __ldcg(reinterpret_cast<const float4 *>(p + kBM * kSplitMaxRows + q));
              u[q] += b.x;
              u[q + 1] += b.y;
              u[q + 2] += b.z;
              u[q + 3] += b.w;
            }
          }
        }
        if (pair) {
          // the two 128-row halves of the W2 block, each its own columns
          emit16(t, n0, t.j * 2 * kBM, g, u);
          emit16(t, n0, t.j * 2 * kBM + kBM, u, g);
        } else {
          emit16(t, n0, t.j * kBM, g, u);
        }
      }
    }
    if (!kGateUp && !(vmax <= 65504.0f)) atomicOr(status, kStatusRange);
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host --

}  // namespace

// Weight map: W viewed as [E][P][rows][K] (P = 2 halves of W13, or 1 for
// W2) with K split into 64-element blocks, the block index ordered after the
// rows: dims {64, rows, P, K/64, E}.  A box [kStageKB][P][box_rows][64] lands
// in shared memory as kStageKB consecutive 128-row K-major tiles.
bool weight_map(CUtensorMap *m, const void *w, int K, int rows, int P, int E, int box_rows) {
  const cuuint64_t dims[5] = {(cuuint64_t)kBK, (cuuint64_t)rows, (cuuint64_t)P,
                              (cuuint64_t)(K / kBK), (cuuint64_t)E};
  const cuuint64_t rs = (cuuint64_t)K * 2;
  const cuuint64_t strides[4] = {rs, rs * rows, (cuuint64_t)kBK * 2, rs * rows * P};
  const cuuint32_t box[5] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, (cuuint32_t)P,
                             (cuuint32_t)kStageKB, 1};
  return encode_bf16_map(m, w, 5, dims, strides, box);
}

// Token rows [R][K] viewed as dims {64, R, K/64}; a box [kblocks][h][64]
// (kblocks = kStageKB unless given).
bool act_map(CUtensorMap *m, const void *a, int K, int64_t R, int box_rows, int kblocks) {
  const cuuint64_t dims[3] = {(cuuint64_t)kBK, (cuuint64_t)R, (cuuint64_t)(K / kBK)};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kBK * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, (cuuint32_t)kblocks};
  return encode_bf16_map(m, a, 3, dims, strides, box);
}

// E4M3 weights [E][P][rows][K] (one byte per weight) as {64, rows, P, K/64,
// E}: a box [kStageKB][P][box_rows][64 bytes], 64-byte swizzled.
bool weight_map_u8(CUtensorMap *m, const void *w, int K, int rows, int P, int E, int box_rows) {
  const cuuint64_t dims[5] = {(cuuint64_t)kBK, (cuuint64_t)rows, (cuuint64_t)P,
                              (cuuint64_t)(K / kBK), (cuuint64_t)E};
  const cuuint64_t rs = (cuuint64_t)K;
  const cuuint64_t strides[4] = {rs, rs * rows, (cuuint64_t)kBK, rs * rows * P};
  const cuuint32_t box[5] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, (cuuint32_t)P,
                             (cuuint32_t)kStageKB, 1};
  return encode_u8_map(m, w, 5, dims, strides, box);
}

namespace {

// The tensor maps of one GEMM launch.  Encoding them takes host time on every
// call (about 20 cuTensorMapEncodeTiled calls per GEMM), so the sets of recent
// calls are kept, keyed by everything the maps depend on: the device, the
// weight and activation pointers and the shapes.
struct GemmMaps {
  CUtensorMap ma, msh, maw, mawsh;
  TokenMaps mb;
};
struct GemmMapKey {
  int dev, E, K, rows, P, shared, pair_maps;
  int64_t R;
  const void *w, *w_sh, *act;
  bool operator==(const GemmMapKey &o) const {
    return dev == o.dev && E == o.E && K == o.K && rows == o.rows && P == o.P &&
           shared == o.shared && pair_maps == o.pair_maps && R == o.R && w == o.w &&
           w_sh == o.w_sh && act == o.act;
  }
};

template <bool kGateUp>
bool encode_gemm_maps(const GemmMapKey &k, GemmMaps *g) {
  // rows of each half of W13 / of W2 per tile; gate/up in the wide layout
  // takes kGateUpColsWide rows of each half
  if (!weight_map(&g->ma, k.w, k.K, k.rows, k.P, k.E, kBM)) return false;
  if (k.shared) {
    if (!weight_map(&g->msh, k.w_sh, k.K, k.rows, k.P, 1, kBM)) return false;
  } else {
    g->msh = g->ma;
  }
  if (kGateUp || k.pair_maps) {
    // gate/up: 64-row boxes (wide layout); down, pair layouts: 256-row boxes
    const int box = kGateUp ? kGateUpColsWide : 2 * kBM;
    if (!weight_map(&g->maw, k.w, k.K, k.rows, k.P, k.E, box)) return false;
    if (k.shared) {
      if (!weight_map(&g->mawsh, k.w_sh, k.K, k.rows, k.P, 1, box)) return false;
    } else {
      g->mawsh = g->maw;
    }
  } else {
    g->maw = g->ma;
    g->mawsh = g->msh;
  }
  for (int i = 0; i < 16; ++i)
    if (!act_map(&g->mb.m[i], k.act, k.K, k.R, 16 * (i + 1))) return false;
  return true;
}

// A small cache of recently used map sets per GEMM kind (round-robin
// replacement); returns false if the encoder rejects the arguments.
template <bool kGateUp>
bool gemm_maps(const GemmMapKey &key, GemmMaps *out) {
  constexpr int kSlots = 16;
  static GemmMapKey keys[kSlots];
  static GemmMaps maps[kSlots];
  static bool used[kSlots] = {};
  static int next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < kSlots; ++i)
    if (used[i] && keys[i] == key) {
      *out = maps[i];
      return true;
    }
  GemmMaps g;
  if (!encode_gemm_maps<kGateUp>(key, &g)) return false;
  keys[next] = key;
  maps[next] = g;
  used[next] = true;
  next = (next + 1) % kSlots;
  *out = g;
  return true;
}

template <bool kGateUp>
cudaError_t launch_gemm(const moe_layer_desc_t &d, const void *w, const void *w_sh,
                        const __nv_bfloat16 *act, const int32_t *plan, int plan_early,
                        const float *w_perm,
                        void *out, float *split_part, uint32_t *split_cnt, uint32_t *status,
                        bool pair_ok, cudaStream_t s) {
  using C = Cfg<kGateUp>;
  const int shared = d.has_shared_expert ? 1 : 0;
  const int nseg = d.E + shared;
  const int64_t Na = (int64_t)d.T * d.k;
  const int64_t R = Na + (shared ? d.T : 0);
  const int K = kGateUp ? d.H : d.I;
  const int rows = kGateUp ? d.I : d.H;  // weight rows per half = output columns
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  GemmMapKey key;
  memset(&key, 0, sizeof key);
  key.dev = dev;
  key.E = d.E;
  key.K = K;
  key.rows = rows;
  key.P = kGateUp ? 2 : 1;
  key.shared = shared;
  key.pair_maps = (!kGateUp && d.H >= 2 * kBM) ? 1 : 0;
  key.R = R;
  key.w = w;
  key.w_sh = shared ? w_sh : nullptr;
  key.act = act;
  GemmMaps g;
  if (!gemm_maps<kGateUp>(key, &g)) return cudaErrorInvalidValue;

  // prefill batches: tiles of 256 weight rows on CTA pairs (the pair kernel
  // reads only the plan's segment rows)
  if (pair_ok && gemm_pair_supported(d, kGateUp))
    return launch_expert_gemm_pair(kGateUp, kGateUp ? g.maw : g.ma, kGateUp ? g.mawsh : g.msh,
                                   g.mb, plan, nseg, d.E, K, rows, Na, w_perm, out, status, s);

  const size_t smem = C::smem_bytes(nseg);
  auto kern = expert_gemm_kernel<kGateUp>;
  static size_t configured[64] = {};  // per device
  if (smem > configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  // one CTA per SM: the device-side plan decides the tiles (and split-K
  // pieces); CTAs without work leave at once
  const int grid = num_sms();
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, g.ma, g.msh, g.maw, g.mawsh, g.mb,
                    plan,
                    plan_early, nseg, d.E, K, rows, Na, w_perm, out, split_part, split_cnt, status);
}

}  // namespace

cudaError_t launch_expert_gateup(const moe_layer_desc_t &d, const void *w13, const void *w13_shared,
                                 const __nv_bfloat16 *x_perm, const int32_t *plan, int plan_early,
                                 float *split_part, uint32_t *split_cnt, __nv_bfloat16 *h,
                                 uint32_t *status, bool pair_ok, cudaStream_t s) {
  return launch_gemm<true>(d, w13, w13_shared, x_perm, plan, plan_early, nullptr, h, split_part,
                           split_cnt, status, pair_ok, s);
}

cudaError_t launch_expert_down(const moe_layer_desc_t &d, const void *w2, const void *w2_shared,
                               const __nv_bfloat16 *h, const int32_t *plan, const float *w_perm,
                               float *split_part, uint32_t *split_cnt, __half *out_perm,
                               uint32_t *status, bool pair_ok, cudaStream_t s) {
  // the plan comes from the dispatch or the gather kernel: at least two
  // launches before the down GEMM
  return launch_gemm<false>(d, w2, w2_shared, h, plan, 1, w_perm, out_perm, split_part, split_cnt,
                            status, pair_ok, s);
}

}  // namespace moe
