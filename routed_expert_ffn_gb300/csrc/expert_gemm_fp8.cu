// Grouped expert GEMMs with FP8 (E4M3) expert weights, for batches above
// the persistent decode layer's 16 tokens ("MoE推理优化全景指南", section
// "量化与 offload 并非独立开关", "专家权重量化": FP8 weights halve the bytes
// the weight-bound expert GEMMs stream).  The two GEMMs of the bf16 chain,
//
//   gate/up:  h[p, i]   = SiLU(sum_c W13[e][i][c] x[p][c]) * sum_c W13[e][I+i][c] x[p][c]
//   down:     out[p, r] = w_perm[p] * sum_i W2[e][r][i] h[p][i]
//
// with W = code * 2^s per 128 x 128 block (exact in fp16), and x_perm and h
// in fp16.  Swap-AB as in the bf16 kernel: weight rows are the MMA's M =
// 128, an expert's token rows (<= 128 per tile) its N.  The weights arrive as
// E4M3 codes by TMA (64-byte swizzled); converter warps turn each K block
// into fp16 values times the block's scale and store them into TMEM, where
// the MMA reads its A operand (tcgen05.mma with A in TMEM); the token rows
// come into shared memory by TMA.  Per weight, shared memory carries the
// copy's byte and the converters' read of it -- against 2 + 2 bytes for bf16
// weights -- so the ring holds eight K blocks of weights in flight.
//
// Tile = (segment, weight block j, 128-row token chunk): gate/up j = 128 h
// columns (their 128 gate rows and 128 up rows, the two halves of the tile),
// down j = 256 W2 rows (two halves of 128).  Tiles of one weight block are
// adjacent (chunk innermost, so CTAs working at the same time share its
// codes through L2); CTA c walks tiles c, c + grid, ...  A K step is two K
// blocks (one staged unit); a K range that ends inside a unit reads zeros.
//
// CTA = 6 warps + the converters:
//   warp 4 lane 0  TMA: each unit's codes (2 K blocks x 2 halves x 128 rows
//                  x 64 bytes) into the four 32 KB staging stages;
//   warp 4 lane 1  TMA: each K block's token rows into one of four operand
//                  stages;
//   warp 5         TMEM (512 columns: one accumulator buffer of 2 x 128
//                  columns, four operand stages of 2 x 32); one thread
//                  issues the MMAs;
//   warps 6-       converters (kFConvSets sets of four), warp w writing the
//                  TMEM lanes of quarter w % 4;
//   warps 0-3      epilogue: SiLU(gate)*up into h, or the gate weighting into
//                  out_perm, both fp16 (saturating at +-65504, which latches
//                  the status word's range bit), then the tile's rows.
// Every wait is bounded; on expiry the CTA latches MOE_ERR_TIMEOUT's status
// bit, leaves its loops, drains its copies and frees TMEM.
#include <cuda_fp8.h>
#include <string.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

// converter sets: each set of four warps converts every kFConvSets-th K block
// of a staged unit (measured with two sets: 0.5-1% slower at every shape;
// building each code's fp16 bits with integer operations instead of the
// conversion instruction: 26-50% slower)
constexpr int kFConvSets = 1;
constexpr int kFThreads = (6 + 4 * kFConvSets) * 32;
constexpr int kFRows = 128;                           // token rows per tile
constexpr uint32_t kFStage = 2 * 2 * kBM * kBK;       // 32 KB of codes per unit
constexpr int kFStages = 4;
constexpr uint32_t kFOpStage = kFRows * kBK * 2;      // 16 KB: <= 128 fp16 token rows
constexpr int kFOpStages = 4;
// one accumulator buffer (a tile's two accumulators of kFRows columns),
// then the operand stages (measured against 64-row tiles with two
// accumulator buffers: Qwen3 T=1024 762 -> 615 us, Mixtral T=512 838 -> 556
// us, DeepSeek-V3 T=2048 4045 -> 3106 us, equal at T <= 128: each expert's
// codes are converted once per 128 token rows instead of 64)
constexpr uint32_t kFAccCols = 2 * kFRows;
constexpr uint32_t kFACol = kFAccCols;
constexpr uint32_t kFAStageCols = 2 * kBK / 2;        // two halves x 32 columns
constexpr uint32_t kFTmemCols = 512;
static_assert(kFACol + kFOpStages * kFAStageCols <= kFTmemCols, "TMEM budget");
static_assert(kStageKB == 2, "a unit is two K blocks");
static_assert(kStageKB % kFConvSets == 0 && kFOpStages % kFConvSets == 0,
              "each converter set owns every kFConvSets-th operand stage");

constexpr size_t fp8_smem_bytes(int nseg) {
  return 1024 + (size_t)kFStages * kFStage + (size_t)kFOpStages * kFOpStage +
         2 * 8 * kBM * 4               // output slices [2][8][128] words
         + kFRows * 4                  // gate weights of a tile
         + (2 * kFStages + 2 * kFOpStages + 5) * 8 + 16 + (size_t)2 * (nseg + 1) * 4;
}
static_assert(fp8_smem_bytes(kMaxE + 1) <= 232448, "shared memory per CTA");

__device__ __forceinline__ void epi_sync_f() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_all_f(bool p) {
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

// D[tmem] (+)= A[tmem] * B[smem]^T: A's rows in the TMEM lanes, two 16-bit
// elements of K per column; fp16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_ts_f16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void kblock_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc) {
  umma_ts_f16(d, a, b, idesc, acc);
  umma_ts_f16(d, a + 8, b + 2, idesc, 1u);
  umma_ts_f16(d, a + 16, b + 4, idesc, 1u);
  umma_ts_f16(d, a + 24, b + 6, idesc, 1u);
}
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&v)[32]) {
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
__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// fp16 x fp16 -> fp32, both K-major
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Two E4M3 codes (the low 16 bits) to two fp16 values times `scale`.
__device__ __forceinline__ uint32_t codes2_to_f16x2(uint32_t two, __half2 scale) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
  const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&hr), scale);
  return *reinterpret_cast<const uint32_t *>(&v);
}

struct FTile {
  int seg, j, row0, nrows;
};

__device__ __forceinline__ FTile fp8_tile(int tile, const int32_t *seg_row, const int32_t *tp,
                                          int nseg) {
  int lo = 0, hi = nseg;  // tp[lo] <= tile < tp[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tp[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  FTile t;
  t.seg = lo;
  const int m = seg_row[lo + 1] - seg_row[lo];
  const int chunks = (m + kFRows - 1) / kFRows;
  const int local = tile - tp[lo];
  t.j = local / chunks;
  const int c = local - t.j * chunks;
  t.row0 = seg_row[lo] + c * kFRows;
  t.nrows = min(kFRows, m - c * kFRows);
  return t;
}

template <bool kGateUp>
__global__ void __launch_bounds__(kFThreads, 1)
    expert_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a,     // codes, routed
                           const __grid_constant__ CUtensorMap tm_a_sh,  // codes, shared expert
                           const __grid_constant__ TokenMaps tm_b,       // fp16 token rows
                           const int8_t *__restrict__ scale, const int8_t *__restrict__ scale_sh,
                           const int32_t *__restrict__ plan, int nseg, int E, int K, int out_cols,
                           int64_t Na, const float *__restrict__ w_perm, uint16_t *__restrict__ out,
                           uint32_t *__restrict__ status) {
  constexpr uint32_t kCode = kGateUp ? kStatusTimeoutGateUp : kStatusTimeoutDown;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *stg = smem;                                                  // [stage][codes]
  uint8_t *opb = stg + kFStages * kFStage;                              // [stage][token rows]
  uint32_t *sOut = reinterpret_cast<uint32_t *>(opb + kFOpStages * kFOpStage);  // [2][8][128]
  float *sW = reinterpret_cast<float *>(sOut + 2 * 8 * kBM);            // [kFRows]
  uint64_t *st_full = reinterpret_cast<uint64_t *>(sW + kFRows);
  uint64_t *st_empty = st_full + kFStages;
  uint64_t *op_full = st_empty + kFStages;
  uint64_t *op_empty = op_full + kFOpStages;
  uint64_t *tfull = op_empty + kFOpStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *fin = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int32_t *seg_row = reinterpret_cast<int32_t *>(tmem_slot + 4);
  int32_t *tp = seg_row + nseg + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kFStages; ++i) {
      mbar_init(&st_full[i], 1);   // the producer's expected bytes
      mbar_init(&st_empty[i], 4 * kFConvSets);  // every converter warp
    }
    for (int i = 0; i < kFOpStages; ++i) {
      mbar_init(&op_full[i], 5);   // token-row copy + four converter warps
      mbar_init(&op_empty[i], 1);  // the MMA's commit
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
    tmem_alloc(tmem_slot, kFTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_sh);
    for (int i = 0; i < kFRows / 16; ++i) tma_prefetch_desc(&tm_b.m[i]);
  }
  pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i <= nseg; i += blockDim.x) seg_row[i] = __ldcg(plan + i);
  __syncthreads();
  // weight blocks per tile row: gate/up 128 h columns, down 256 W2 rows
  const int nj = kGateUp ? (out_cols + kBM - 1) / kBM : (out_cols + 2 * kBM - 1) / (2 * kBM);
  if (warp == 0) {
    const int per = (nseg + 31) / 32;
    const int s0 = lane * per, s1 = min(nseg, s0 + per);
    int sum = 0;
    for (int s = s0; s < s1; ++s) sum += (seg_row[s + 1] - seg_row[s] + kFRows - 1) / kFRows * nj;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int s = s0; s < s1; ++s) {
      tp[s] = run;
      run += (seg_row[s + 1] - seg_row[s] + kFRows - 1) / kFRows * nj;
    }
    if (lane == 31) tp[nseg] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tp[nseg];
  const int nkb = K / kBK;
  const int nu = (nkb + kStageKB - 1) / kStageKB;  // units (K steps) per tile
  // 128 x 128 scale blocks: rows (per half of W13, or of W2) and K
  const int nrb = kGateUp ? (out_cols + kBM - 1) / kBM : (out_cols + kBM - 1) / kBM;
  const int nkb128 = (K + kBM - 1) / kBM;

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------ TMA: weight codes --
      uint32_t st = 0, ph = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const FTile t = fp8_tile(tile, seg_row, tp, nseg);
        const bool sh = t.seg >= E;
        const CUtensorMap *ma = sh ? &tm_a_sh : &tm_a;
        const int ecoord = sh ? 0 : t.seg;
        const int arow = kGateUp ? t.j * kBM : t.j * 2 * kBM;
        for (int v = 0; v < nu; ++v) {
          if (!mbar_wait(&st_empty[st], ph ^ 1u, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&st_full[st], kFStage);
          tma_load_5d(stg + st * kFStage, ma, &st_full[st], 0, arow, 0, kStageKB * v, ecoord);
          ++issued;
          if (++st == (uint32_t)kFStages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      const uint32_t n = issued < (uint32_t)kFStages ? issued : (uint32_t)kFStages;
      for (uint32_t i = 0; i < n; ++i) {
        st = st == 0 ? kFStages - 1 : st - 1;
        if (st == (uint32_t)kFStages - 1) ph ^= 1u;
        mbar_wait_drain(&st_full[st], ph);
      }
    } else if (lane == 1) {
      // ------------------------------------------------- TMA: token rows --
      uint32_t st = 0, ph = 0, issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const FTile t = fp8_tile(tile, seg_row, tp, nseg);
        const int n16 = (t.nrows + 15) & ~15;
        const CUtensorMap *mb = &tm_b.m[(n16 >> 4) - 1];
        for (int kb = 0; kb < kStageKB * nu; ++kb) {
          if (!mbar_wait(&op_empty[st], ph ^ 1u, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&op_full[st], (uint32_t)n16 * (kBK * 2));
          tma_load_3d(opb + st * kFOpStage, mb, &op_full[st], 0, t.row0, kb);
          ++issued;
          if (++st == (uint32_t)kFOpStages) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      const uint32_t n = issued < (uint32_t)kFOpStages ? issued : (uint32_t)kFOpStages;
      for (uint32_t i = 0; i < n; ++i) {
        st = st == 0 ? kFOpStages - 1 : st - 1;
        if (st == (uint32_t)kFOpStages - 1) ph ^= 1u;
        mbar_wait_drain(&op_full[st], ph);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t st = 0, ph = 0, tl = 0;
      const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(opb));
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++tl) {
        const FTile t = fp8_tile(tile, seg_row, tp, nseg);
        const int n16 = (t.nrows + 15) & ~15;
        const uint32_t id = idesc_f16(kBM, n16);
        const uint32_t buf = 0u, use = tl;  // one accumulator buffer
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, status, kCode)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * kFAccCols;
        for (int kb = 0; kb < kStageKB * nu; ++kb) {
          if (!mbar_wait(&op_full[st], ph, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bdesc = bdesc0 + st * (kFOpStage >> 4);
          const uint32_t a0 = tmem_base + kFACol + st * kFAStageCols;
          const uint32_t acc = kb != 0 ? 1u : 0u;
          // gate/up: gate rows, up rows; down: W2 rows [0,128), [128,256)
          kblock_ts(d0, a0, bdesc, id, acc);
          kblock_ts(d0 + kFRows, a0 + kFAStageCols / 2, bdesc, id, acc);
          umma_commit(&op_empty[st]);  // operand stage free once these MMAs have read it
          if (++st == (uint32_t)kFOpStages) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[buf]);
      }
      umma_commit(fin);
      mbar_wait_drain(fin, 0);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------------------------------------------------- converters --
    // Each K block of a staged unit: the two 128-row halves (128 rows x 64
    // codes) become 128 rows x 64 fp16 times the block's scale in the
    // operand stage's TMEM columns.  One weight row per thread: the row's 64
    // codes are four 16-byte chunks read through the 64-byte swizzle (the
    // warp's 32 rows touch every bank once per phase).
    const int quarter = warp & 3;
    const int cset = (warp - 6) >> 2;   // this warp's converter set
    const int r = quarter * 32 + lane;  // weight row of a half
    const int sw = (r >> 1) & 3;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16) + kFACol;
    uint32_t s1 = 0, p1 = 0, s2 = (uint32_t)cset, p2 = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const FTile t = fp8_tile(tile, seg_row, tp, nseg);
      const bool sh = t.seg >= E;
      const int8_t *sc = sh ? scale_sh : scale;
      const int ex = sh ? 0 : t.seg;
      for (int v = 0; ok && v < nu; ++v) {
        __half2 scl[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // gate/up: [E][2][nrb][nkb128] (half = gate / up); down:
          // [E][nrb][nkb128] (half = row block 2j + half); a row block past
          // the matrix holds zero codes
          int e8 = 0;
          if (kGateUp) {
            e8 = sc[((ex * 2 + half) * nrb + t.j) * nkb128 + v];
          } else if (2 * t.j + half < nrb) {
            e8 = sc[(ex * nrb + 2 * t.j + half) * nkb128 + v];
          }
          scl[half] = __float2half2_rn(ldexpf(1.0f, e8));  // 2^e8, exact in fp16
        }
        if (!mbar_wait(&st_full[s1], p1, abort_flag, status, kCode)) {
          ok = false;
          break;
        }
        const uint8_t *src = stg + s1 * kFStage;
        for (int hk = cset; hk < kStageKB; hk += kFConvSets) {
          if (!mbar_wait(&op_empty[s2], p2 ^ 1u, abort_flag, status, kCode)) {
            ok = false;
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
                w[8 * c + 2 * q] = codes2_to_f16x2(wd[q], scl[half]);
                w[8 * c + 2 * q + 1] = codes2_to_f16x2(wd[q] >> 16, scl[half]);
              }
            }
            tmem_store32(lane_base + s2 * kFAStageCols + half * (kFAStageCols / 2), w);
          }
          tmem_store_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&op_full[s2]);
          s2 += kFConvSets;
          if (s2 >= (uint32_t)kFOpStages) {
            s2 -= kFOpStages;
            p2 ^= 1u;
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&st_empty[s1]);
        if (++s1 == (uint32_t)kFStages) {
          s1 = 0;
          p1 ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    // Per 16-token slice: tcgen05.ld of the thread's row in both halves, the
    // fused math, two tokens per conversion into words [8 token pairs][128
    // columns] in shared memory, then every thread stores 16 bytes of a
    // token pair's rows (the pairs split by byte permutes).
    const int r = warp * 32 + lane;
    uint32_t tl = 0, slice = 0;
    float vmax = 0.f;  // the largest magnitude of a stored value (NaN-propagating)
    auto emit = [&](const FTile &t, int n0, int col0, const uint32_t (&word)[8]) {
      uint32_t *so = sOut + (slice & 1u) * (8 * kBM);
#pragma unroll
      for (int p = 0; p < 8; ++p) so[p * kBM + r] = word[p];
      epi_sync_f();
      const int p = r >> 4, ch = r & 15;
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
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tl) {
      const FTile t = fp8_tile(tile, seg_row, tp, nseg);
      const uint32_t buf = 0u, use = tl;
      const bool waited = mbar_wait(&tfull[buf], use & 1u, abort_flag, status, kCode);
      if (!epi_all_f(waited && !*abort_flag)) break;
      tc_fence_after();
      if (!kGateUp) {
        if (r < kFRows) {
          const int64_t row = (int64_t)t.row0 + r;
          sW[r] = (r < t.nrows && w_perm != nullptr && t.seg < E && row < Na) ? w_perm[row] : 1.0f;
        }
        epi_sync_f();
      }
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + buf * kFAccCols;
      const int N = (t.nrows + 15) & ~15;
      for (int n0 = 0; n0 < N; n0 += 16) {
        if (kGateUp) {
          uint32_t g0[16], u0[16];
          tmem_ld16(tb + n0, g0);
          tmem_ld16(tb + kFRows + n0, u0);
          tmem_ld_wait();
          uint32_t word[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float ga = __uint_as_float(g0[2 * p]), gb = __uint_as_float(g0[2 * p + 1]);
            const float ha = __fdividef(ga, 1.0f + __expf(-ga)) * __uint_as_float(u0[2 * p]);
            const float hb = __fdividef(gb, 1.0f + __expf(-gb)) * __uint_as_float(u0[2 * p + 1]);
            // only the tile's own token columns count towards the range check
            vmax = fmax_nan(vmax, n0 + 2 * p < t.nrows ? fabsf(ha) : 0.f);
            vmax = fmax_nan(vmax, n0 + 2 * p + 1 < t.nrows ? fabsf(hb) : 0.f);
            word[p] = pack_f16x2_satfinite(ha, hb);
          }
          emit(t, n0, t.j * kBM, word);
        } else {
          float wv[16];
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(sW + n0 + q);
            wv[q] = a4.x;
            wv[q + 1] = a4.y;
            wv[q + 2] = a4.z;
            wv[q + 3] = a4.w;
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v0[16];
            tmem_ld16(tb + hh * kFRows + n0, v0);
            tmem_ld_wait();
            uint32_t word[8];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const float xa = __uint_as_float(v0[2 * p]) * wv[2 * p];
              const float xb = __uint_as_float(v0[2 * p + 1]) * wv[2 * p + 1];
              vmax = fmax_nan(vmax, n0 + 2 * p < t.nrows ? fabsf(xa) : 0.f);
              vmax = fmax_nan(vmax, n0 + 2 * p + 1 < t.nrows ? fabsf(xb) : 0.f);
              word[p] = pack_f16x2_satfinite(xa, xb);
            }
            emit(t, n0, t.j * 2 * kBM + hh * kBM, word);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
    if (!(vmax <= 65504.0f)) atomicOr(status, kStatusRange);
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kFTmemCols);
  }
}

// The tensor maps of one FP8 GEMM launch, cached like the bf16 GEMM's.
struct Fp8Maps {
  CUtensorMap ma, msh;
  TokenMaps mb;
};
struct Fp8Key {
  int dev, gate_up, E, K, rows, shared;
  int64_t R;
  const void *w, *w_sh, *act;
  bool operator==(const Fp8Key &o) const {
    return dev == o.dev && gate_up == o.gate_up && E == o.E && K == o.K && rows == o.rows &&
           shared == o.shared && R == o.R && w == o.w && w_sh == o.w_sh && act == o.act;
  }
};

bool fp8_maps(const Fp8Key &k, Fp8Maps *out) {
  constexpr int kSlots = 16;
  static Fp8Key keys[kSlots];
  static Fp8Maps maps[kSlots];
  static bool used[kSlots] = {};
  static int next = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < kSlots; ++i)
    if (used[i] && keys[i] == k) {
      *out = maps[i];
      return true;
    }
  Fp8Maps m;
  memset(&m, 0, sizeof m);
  // gate/up: 128 gate + 128 up rows (P = 2); down: 256 W2 rows
  const int P = k.gate_up ? 2 : 1, box = k.gate_up ? kBM : 2 * kBM;
  if (!weight_map_u8(&m.ma, k.w, k.K, k.rows, P, k.E, box)) return false;
  if (k.shared) {
    if (!weight_map_u8(&m.msh, k.w_sh, k.K, k.rows, P, 1, box)) return false;
  } else {
    m.msh = m.ma;
  }
  for (int i = 0; i < kFRows / 16; ++i)
    if (!act_map(&m.mb.m[i], k.act, k.K, k.R, 16 * (i + 1), 1)) return false;
  for (int i = kFRows / 16; i < 16; ++i) m.mb.m[i] = m.mb.m[0];
  keys[next] = k;
  maps[next] = m;
  used[next] = true;
  next = (next + 1) % kSlots;
  *out = m;
  return true;
}

}  // namespace

cudaError_t launch_expert_gemm_fp8(bool gate_up, const moe_layer_desc_t &d, const void *w,
                                   const int8_t *w_scale, const void *w_sh,
                                   const int8_t *w_sh_scale, const void *act,
                                   const int32_t *plan, const float *w_perm, void *out,
                                   uint32_t *status, cudaStream_t s) {
  const int shared = d.has_shared_expert ? 1 : 0;
  const int nseg = d.E + shared;
  const int64_t Na = (int64_t)d.T * d.k;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  Fp8Key key;
  memset(&key, 0, sizeof key);
  key.dev = dev;
  key.gate_up = gate_up ? 1 : 0;
  key.E = d.E;
  key.K = gate_up ? d.H : d.I;
  key.rows = gate_up ? d.I : d.H;
  key.shared = shared;
  key.R = Na + (shared ? d.T : 0);
  key.w = w;
  key.w_sh = shared ? w_sh : nullptr;
  key.act = act;
  Fp8Maps m;
  if (!fp8_maps(key, &m)) return cudaErrorInvalidValue;
  const size_t smem = fp8_smem_bytes(nseg);
  auto kern = gate_up ? expert_gemm_fp8_kernel<true> : expert_gemm_fp8_kernel<false>;
  static size_t configured[2][64] = {};
  const int g = gate_up ? 1 : 0;
  if (smem > configured[g][dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[g][dev] = smem;
  }
  return launch_pdl(kern, dim3(num_sms()), dim3(kFThreads), smem, s, m.ma, m.msh, m.mb, w_scale,
                    shared ? w_sh_scale : w_scale, plan, nseg, d.E, key.K, key.rows, Na, w_perm,
                    static_cast<uint16_t *>(out), status);
}

}  // namespace moe
