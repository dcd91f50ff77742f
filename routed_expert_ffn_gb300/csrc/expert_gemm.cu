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
// the expert's token rows its N dimension (16..128, rounded up to 16).  In
// the decode regime an expert sees only a handful of rows, yet every weight
// byte is read from HBM once per (expert, 128-row token chunk) and streamed
// through the tensor cores at full M; in the prefill regime tiles are full
// 128 x 128.
//
// Work unit (tile) = (segment s, weight-row block j, token chunk c); segments
// are the E experts (+ the shared expert, all T tokens).  The tile plan (a
// prefix sum of tiles per segment, computed on the device from the dispatch
// offsets) is read by a persistent kernel, one CTA per SM, which walks tiles
// blockIdx.x, blockIdx.x + gridDim.x, ...  Tiles of one weight block are
// adjacent (chunk index innermost) so CTAs working at the same time share
// weight tiles through L2; experts with no rows have no tiles, so their
// weights are never read.
//
// CTA = 6 warps:
//   warp 4      TMA producer: weight tile(s) [128 x 64] and token tile
//               [16-row boxes x 64] per K step into a STAGES-deep ring
//               (128-byte swizzle), completion on the stage's mbarrier;
//   warp 5      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma (bf16 in, fp32 accumulate in TMEM), commits the
//               stage back to the producer and the finished accumulator to
//               the epilogue; two accumulator buffers let the epilogue of one
//               tile overlap the mainloop of the next;
//   warps 0-3   epilogue: tcgen05.ld of their 32 TMEM lanes (= 32 weight
//               rows), fused SiLU(gate)*up (gate/up GEMM) or gate weighting
//               (down GEMM), bf16 (h) or fp16 (out_perm) stores.
// Every wait is bounded; on expiry the CTA records MOE_ERR_TIMEOUT's status
// bit, drains its copies and MMAs in flight, frees TMEM and returns.
#include <stdio.h>

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


namespace {

constexpr int kThreads = 192;
constexpr int kStagesGateUp = MOE_STAGES_GATEUP;
constexpr int kStagesDown = MOE_STAGES_DOWN;

__host__ __device__ constexpr uint32_t tmem_cols_pow2(uint32_t n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

template <bool kGateUp, int BN, int STAGES>
struct Cfg {
  static constexpr int NA = kGateUp ? 2 : 1;               // weight tiles per stage
  static constexpr uint32_t A_BYTES = kBM * kBK * 2;       // 16 KB
  static constexpr uint32_t B_BYTES = BN * kBK * 2;        // BN rows of 128 B
  static constexpr uint32_t B16_BYTES = 16 * kBK * 2;      // one 16-row box
  static constexpr uint32_t STAGE_BYTES = NA * A_BYTES + B_BYTES;
  static constexpr uint32_t ACC_COLS = NA * BN;            // TMEM columns per tile
  static constexpr uint32_t TMEM_COLS = tmem_cols_pow2(2 * ACC_COLS);
  static constexpr uint32_t BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
  static constexpr uint32_t STAGE_OUT_BYTES = 16 * kBM * 2;  // one 16-token output slice
  static size_t smem_bytes(int nseg) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + STAGE_OUT_BYTES + (size_t)BN * 4 + BAR_BYTES +
           (size_t)2 * (nseg + 1) * 4;
  }
  static_assert(2 * ACC_COLS <= 512, "accumulators exceed TMEM");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "bad token tile");
};

struct Tile {
  int seg, j, row0, nrows;
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

template <int BN>
__device__ __forceinline__ Tile decode_tile(int tile, const int32_t *seg_row, const int32_t *pref,
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
  const int chunks = (m + BN - 1) / BN;
  t.j = local / chunks;
  const int c = local - t.j * chunks;
  t.row0 = seg_row[lo] + c * BN;
  t.nrows = min(BN, m - c * BN);
  return t;
}

template <bool kGateUp, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,     // routed weights (4D)
                       const __grid_constant__ CUtensorMap tm_a_sh,  // shared-expert weights (4D)
                       const __grid_constant__ CUtensorMap tm_b,     // activations [R, K] (2D)
                       const int32_t *__restrict__ plan, int nseg, int E, int K, int out_cols,
                       int64_t Na, const float *__restrict__ w_perm, void *__restrict__ out_,
                       float *__restrict__ split_part, uint32_t *__restrict__ split_cnt,
                       uint32_t *__restrict__ status) {
  using C = Cfg<kGateUp, BN, STAGES>;
  // gate/up writes h in bf16 (the next GEMM's operand); down writes the
  // gate-weighted rows in fp16: 11 significant bits (8x finer than bf16) at
  // the same bandwidth; magnitudes past the fp16 range are clamped and
  // latched in the status word.  Both are 2-byte elements.
  uint16_t *out = static_cast<uint16_t *>(out_);
  constexpr uint32_t kCode = kGateUp ? kStatusTimeoutGateUp : kStatusTimeoutDown;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;                                  // [STAGES][NA][A_BYTES]
  uint8_t *sB = sA + (size_t)STAGES * C::NA * C::A_BYTES;  // [STAGES][B_BYTES]
  uint16_t *sOut = reinterpret_cast<uint16_t *>(sB + (size_t)STAGES * C::B_BYTES);  // [16][kBM]
  float *sW = reinterpret_cast<float *>(sOut + 16 * kBM);  // [BN] gate weights (down)
  uint64_t *full = reinterpret_cast<uint64_t *>(sW + BN);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *fin = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *s_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);  // last split piece
  int *s_split = reinterpret_cast<int *>(tmem_slot + 3);                   // split-K factor
  int32_t *seg_row = reinterpret_cast<int32_t *>(tmem_slot + 4);
  int32_t *pref = seg_row + nseg + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
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
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_a_sh);
    tma_prefetch_desc(&tm_b);
  }
  // everything above is independent of earlier kernels' outputs
  pdl_wait();
  pdl_launch_dependents();
  const int32_t *g_pref = plan + (kGateUp ? 1 : 2) * (nseg + 1);
  for (int i = threadIdx.x; i <= nseg; i += blockDim.x) {
    seg_row[i] = plan[i];
    pref[i] = g_pref[i];
  }
  if (threadIdx.x == 0) *s_split = plan[3 * (nseg + 1) + (kGateUp ? 0 : 1)];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = pref[nseg];
  const int nkb = K / kBK;
  // work unit = one K piece of a tile (S == 1: the whole tile)
  const int S = *s_split;
  const int kbs = (nkb + S - 1) / S;
  const int total_pieces = total * S;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int pc = blockIdx.x; ok && pc < total_pieces; pc += gridDim.x) {
        const int tile = pc / S, z = pc - tile * S;
        const Tile t = decode_tile<BN>(tile, seg_row, pref, nseg);
        const int kb0 = z * kbs, kb1 = min(nkb, kb0 + kbs);
        const bool sh = (t.seg >= E);
        const CUtensorMap *ma = sh ? &tm_a_sh : &tm_a;
        const int ecoord = sh ? 0 : t.seg;
        const int nb16 = (t.nrows + 15) >> 4;
        const uint32_t bytes = C::NA * C::A_BYTES + (uint32_t)nb16 * C::B16_BYTES;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int st = (int)(it % STAGES);
          const uint32_t ph = (it / STAGES) & 1u;
          if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], bytes);
          uint8_t *a0 = sA + (size_t)st * C::NA * C::A_BYTES;
          tma_load_4d(a0, ma, &full[st], kb * kBK, t.j * kBM, 0, ecoord);
          if (kGateUp) tma_load_4d(a0 + C::A_BYTES, ma, &full[st], kb * kBK, t.j * kBM, 1, ecoord);
          uint8_t *b0 = sB + (size_t)st * C::B_BYTES;
          for (int q = 0; q < nb16; ++q)
            tma_load_2d(b0 + q * C::B16_BYTES, &tm_b, &full[st], kb * kBK, t.row0 + q * 16);
        }
      }
      // Drain: every issued copy must land before the CTA may exit.
      const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
      for (uint32_t i = first; i < it; ++i) mbar_wait_drain(&full[i % STAGES], (i / STAGES) & 1u);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int pc = blockIdx.x; ok && pc < total_pieces; pc += gridDim.x, ++tl) {
        const int tile = pc / S, z = pc - tile * S;
        const Tile t = decode_tile<BN>(tile, seg_row, pref, nseg);
        const int kb0 = z * kbs, kb1 = min(nkb, kb0 + kbs);
        const int N = (t.nrows + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(kBM, N);
        const uint32_t buf = tl & 1u, use = tl >> 1;
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, status, kCode)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * C::ACC_COLS;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int st = (int)(it % STAGES);
          if (!mbar_wait(&full[st], (it / STAGES) & 1u, abort_flag, status, kCode)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + (size_t)st * C::NA * C::A_BYTES);
          const uint32_t b_addr = smem_u32(sB + (size_t)st * C::B_BYTES);
          const uint64_t adesc = sdesc_k_sw128(a_addr);
          const uint64_t bdesc = sdesc_k_sw128(b_addr);
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            // advance 16 bf16 (32 bytes) along K inside the swizzled row
            const uint32_t acc = (kb != kb0 || ks != 0) ? 1u : 0u;
            umma_bf16(d0, adesc + 2 * ks, bdesc + 2 * ks, idesc, acc);
            if (kGateUp) {
              const uint64_t adesc_up = sdesc_k_sw128(a_addr + C::A_BYTES);
              umma_bf16(d0 + BN, adesc_up + 2 * ks, bdesc + 2 * ks, idesc, acc);
            }
          }
          umma_commit(&empty[st]);  // stage free once these MMAs have read it
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
    // Per 16-token slice: tcgen05.ld of the thread's weight row (16 token
    // columns), fused SiLU(gate)*up or gate weighting, the slice written
    // transposed into smem, then stored as token rows with 16-byte vector
    // stores by all 128 epilogue threads.  A split-K piece instead writes its
    // fp32 partial; the last piece of the tile adds the S partials in split
    // order and runs the same epilogue.
    const int r = warp * 32 + lane;  // TMEM lane = weight row of the tile
    uint32_t tl = 0;
    bool range_bad = false;
    auto emit16 = [&](const Tile &t, int n0, const float(&g)[16], const float(&u)[16]) {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        uint16_t bits;
        if (kGateUp) {
          bits = __bfloat16_as_ushort(__float2bfloat16_rn(g[q] / (1.0f + __expf(-g[q])) * u[q]));
        } else {
          const float val = g[q] * sW[n0 + q];
          range_bad |= !(fabsf(val) <= 65504.0f);
          bits = __half_as_ushort(__float2half_rn(fminf(fmaxf(val, -65504.0f), 65504.0f)));
        }
        sOut[q * kBM + r] = bits;
      }
      epi_sync();
      // 16 token rows x 128 columns x 2 bytes = 256 chunks of 16 bytes
      const int col0 = t.j * kBM;
      for (int c = r; c < 16 * (kBM / 8); c += 128) {
        const int q = c / (kBM / 8), ch = c % (kBM / 8);
        const int n = n0 + q, col = col0 + ch * 8;
        if (n < t.nrows && col < out_cols)
          *reinterpret_cast<uint4 *>(out + ((int64_t)t.row0 + n) * out_cols + col) =
              *reinterpret_cast<const uint4 *>(sOut + q * kBM + ch * 8);
      }
      epi_sync();
    };
    constexpr int kSlot = C::NA * kBM * kSplitMaxRows;  // floats of one piece's partial
    for (int pc = blockIdx.x; pc < total_pieces; pc += gridDim.x, ++tl) {
      const int tile = pc / S, z = pc - tile * S;
      const Tile t = decode_tile<BN>(tile, seg_row, pref, nseg);
      const uint32_t buf = tl & 1u, use = tl >> 1;
      const bool waited = mbar_wait(&tfull[buf], use & 1u, abort_flag, status, kCode);
      // one decision for all 128 epilogue threads: they share named barriers
      if (!epi_all(waited && !*abort_flag)) break;
      tc_fence_after();
      if (!kGateUp) {
        for (int n = r; n < BN; n += 128) {
          const int64_t row = (int64_t)t.row0 + n;
          sW[n] = (n < t.nrows && w_perm != nullptr && row < Na) ? w_perm[row] : 1.0f;
        }
        epi_sync();
      }
      const uint32_t tb = tmem_base + ((uint32_t)(warp * 32) << 16) + buf * C::ACC_COLS;
      const int N = (t.nrows + 15) & ~15;
      if (S == 1) {
        for (int n0 = 0; n0 < N; n0 += 16) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tb + n0, v0);
          if (kGateUp) tmem_ld16(tb + BN + n0, v1);
          tmem_ld_wait();
          float g[16], u[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            g[q] = __uint_as_float(v0[q]);
            u[q] = kGateUp ? __uint_as_float(v1[q]) : 0.f;
          }
          emit16(t, n0, g, u);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        continue;
      }
      // ---- split-K piece (N <= kSplitMaxRows): fp32 partial to global ----
      float *slot = split_part + (size_t)(tile * S + z) * kSlot + (size_t)r * kSplitMaxRows;
      for (int n0 = 0; n0 < N; n0 += 16) {
        uint32_t v0[16], v1[16];
        tmem_ld16(tb + n0, v0);
        if (kGateUp) tmem_ld16(tb + BN + n0, v1);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 16; q += 4) {
          *reinterpret_cast<float4 *>(slot + n0 + q) =
              make_float4(__uint_as_float(v0[q]), __uint_as_float(v0[q + 1]),
                          __uint_as_float(v0[q + 2]), __uint_as_float(v0[q + 3]));
          if (kGateUp)
            *reinterpret_cast<float4 *>(slot + kBM * kSplitMaxRows + n0 + q) =
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
              split_part + (size_t)(tile * S + zz) * kSlot + (size_t)r * kSplitMaxRows + n0;
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(p + q));
            g[q] += a.x;
            g[q + 1] += a.y;
            g[q + 2] += a.z;
            g[q + 3] += a.w;
            if (kGateUp) {
              const float4 b = __ldcg(reinterpret_cast<const float4 *>(p + kBM * kSplitMaxRows + q));
              u[q] += b.x;
              u[q + 1] += b.y;
              u[q + 2] += b.z;
              u[q + 3] += b.w;
            }
          }
        }
        emit16(t, n0, g, u);
      }
    }
    if (range_bad) atomicOr(status, kStatusRange);
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host --

// Weight map viewed as [E][P][rows][K] (P = 2 halves of W13, or 1 for W2).
bool weight_map(CUtensorMap *m, const void *w, int K, int rows, int P, int E) {
  const cuuint64_t dims[4] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)P, (cuuint64_t)E};
  const cuuint64_t rs = (cuuint64_t)K * 2;
  const cuuint64_t strides[3] = {rs, rs * rows, rs * rows * P};
  const cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)kBM, 1, 1};
  return encode_bf16_map(m, w, 4, dims, strides, box);
}

bool act_map(CUtensorMap *m, const void *a, int K, int64_t R) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)R};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, 16};
  return encode_bf16_map(m, a, 2, dims, strides, box);
}

template <bool kGateUp, int BN, int STAGES>
cudaError_t launch_gemm(const moe_layer_desc_t &d, const void *w, const void *w_sh,
                        const __nv_bfloat16 *act, const int32_t *plan, const float *w_perm,
                        void *out, float *split_part, uint32_t *split_cnt, uint32_t *status,
                        cudaStream_t s) {
  using C = Cfg<kGateUp, BN, STAGES>;
  static_assert(BN == (kGateUp ? kBNGateUp : kBNDown), "the tile plan's token chunks");
  const int shared = d.has_shared_expert ? 1 : 0;
  const int nseg = d.E + shared;
  const int64_t Na = (int64_t)d.T * d.k;
  const int64_t R = Na + (shared ? d.T : 0);
  const int K = kGateUp ? d.H : d.I;
  const int rows = kGateUp ? d.I : d.H;  // weight rows per half = output columns
  const int P = kGateUp ? 2 : 1;
  CUtensorMap ma, msh, mb;
  if (!weight_map(&ma, w, K, rows, P, d.E)) return cudaErrorInvalidValue;
  if (shared) {
    if (!weight_map(&msh, w_sh, K, rows, P, 1)) return cudaErrorInvalidValue;
  } else {
    msh = ma;
  }
  if (!act_map(&mb, act, K, R)) return cudaErrorInvalidValue;

  const size_t smem = C::smem_bytes(nseg);
  auto kern = expert_gemm_kernel<kGateUp, BN, STAGES>;
  static size_t configured[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  // one CTA per SM: the device-side plan decides the tiles (and split-K
  // pieces); CTAs without work leave at once
  const int grid = num_sms();
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, ma, msh, mb, plan, nseg, d.E, K, rows,
                    Na, w_perm, out, split_part, split_cnt, status);
}

}  // namespace

cudaError_t launch_expert_gateup(const moe_layer_desc_t &d, const void *w13, const void *w13_shared,
                                 const __nv_bfloat16 *x_perm, const int32_t *plan,
                                 float *split_part, uint32_t *split_cnt, __nv_bfloat16 *h,
                                 uint32_t *status, cudaStream_t s) {
  return launch_gemm<true, kBNGateUp, kStagesGateUp>(d, w13, w13_shared, x_perm, plan, nullptr, h,
                                                     split_part, split_cnt, status, s);
}

cudaError_t launch_expert_down(const moe_layer_desc_t &d, const void *w2, const void *w2_shared,
                               const __nv_bfloat16 *h, const int32_t *plan, const float *w_perm,
                               float *split_part, uint32_t *split_cnt, __half *out_perm,
                               uint32_t *status, cudaStream_t s) {
  return launch_gemm<false, kBNDown, kStagesDown>(d, w2, w2_shared, h, plan, w_perm, out_perm,
                                                  split_part, split_cnt, status, s);
}

}  // namespace moe
