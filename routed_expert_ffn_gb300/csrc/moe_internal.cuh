// Internal declarations of the sm_103a MoE FFN library: workspace layout,
// launch helpers and the inline-PTX wrappers (mbarrier, TMA, tcgen05) the
// kernels are written with.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------ constants --

constexpr int kMaxE = 512;          // routed experts
constexpr int kMaxK = 32;           // experts per token
constexpr int kMaxT = 1 << 20;
constexpr int64_t kMaxAssign = 1 << 24;

// Router: at most this many K splits (summed by the gating kernel); batches of
// up to kSmallRouteT tokens take the one-launch small-batch router.
constexpr int kRouteMaxSplits = 32;
constexpr int kSmallRouteT = 32;

// The workspace starts with a status block zeroed by moe_workspace_init:
// 32-bit words [0, 64) hold the status word and the small-batch router's
// arrival counter; then 2 x kMaxSplitTiles split-K arrival counters (gate/up,
// down).  Every counter returns to zero when its kernel completes.
constexpr int kRouteCounterWord = 16;  // small-batch router: CTAs finished
constexpr int kSplitCounterWord = 64;  // first split-K counter

// Dispatch: threads per block; each block takes a chunk of the assignment
// list (a multiple of the block size, chosen so there are at most
// kDispatchMaxBlocks blocks).
constexpr int kDispatchThreads = 256;
// (measured: raising it to 8192 made the dispatch 23 us slower at
// T*k = 8192, where three launches overlap through PDL)
#ifndef MOE_SMALL_DISPATCH
#define MOE_SMALL_DISPATCH 2048
#endif
constexpr int64_t kSmallDispatch = MOE_SMALL_DISPATCH;  // N_a up to this: one-block dispatch
constexpr int kDispatchMaxBlocks = 1024;
inline int64_t dispatch_chunk(int64_t Na) {
  int64_t c = (Na + kDispatchMaxBlocks - 1) / kDispatchMaxBlocks;
  c = (c + kDispatchThreads - 1) / kDispatchThreads * kDispatchThreads;
  return c < kDispatchThreads ? kDispatchThreads : c;
}

// Expert GEMMs (tcgen05), stepped through K in blocks of kBK, kStageKB blocks
// per pipeline stage, in one of two layouts chosen per launch by the tile
// plan.  Narrow (most token chunks <= 128 rows): gate/up tile = 128 gate rows
// and the same 128 up rows of W13 by <= kTileRowsGateUp token rows; down tile
// = 128 rows of W2 by <= kTileRowsDown token rows, run one 128-row half per
// stage.  Wide: gate/up tile = kGateUpColsWide gate + the same up rows by
// <= kTileRowsDown token rows; down tile as above in one stage.
constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kTileRowsGateUp = 128;
constexpr int kTileRowsDown = 256;
constexpr int kGateUpColsWide = 64;
// In the narrow gate/up layout, segments of more than this many rows still take
// wide tiles (their stages are the same size).
#ifndef MOE_GU_WIDE_ABOVE
#define MOE_GU_WIDE_ABOVE 1024
#endif
constexpr int kGateUpWideAbove = MOE_GU_WIDE_ABOVE;
#ifndef MOE_STAGE_KB
#define MOE_STAGE_KB 2
#endif
constexpr int kStageKB = MOE_STAGE_KB;
// The down GEMM's "pair" layout: where it would otherwise run narrow, tiles
// of 256 W2 rows (two 128-row halves, two MMAs sharing the token operand) by
// <= 128 token rows: 64 KB of weights per 96 KB stage instead of 32 of 64.
#ifndef MOE_DOWN_PAIR
#define MOE_DOWN_PAIR 1
#endif
constexpr bool kDownPair = MOE_DOWN_PAIR != 0;
// The same pairing in the thin (decode) layout: stages of 64 KB of weights
// + 16 token rows, three in flight (192 KB of weights instead of 160).
#ifndef MOE_DOWN_THIN_PAIR
#define MOE_DOWN_THIN_PAIR 1
#endif
constexpr bool kDownThinPair = MOE_DOWN_THIN_PAIR != 0;
constexpr int kThinRows = 16;           // the thin layout: tiles of <= 16 token rows
constexpr int kMediumRows = 64;         // the down GEMM's medium layout: <= 64 rows
constexpr int kRingBytes = 204 * 1024;  // 3 thin gate/up stages of 68 KB

// Status word bits (latched with atomicOr).
constexpr uint32_t kStatusBadExpertId = 1u << 0;
constexpr uint32_t kStatusTimeoutGateUp = 1u << 1;
constexpr uint32_t kStatusTimeoutDown = 1u << 2;
constexpr uint32_t kStatusBadOffsets = 1u << 3;
constexpr uint32_t kStatusTimeoutRouter = 1u << 4;
constexpr uint32_t kStatusRange = 1u << 5;  // a gate-weighted expert output beyond fp16 range
constexpr uint32_t kStatusTimeoutCheck = 1u << 6;  // the bounded-wait check ran out (expected)
constexpr uint32_t kStatusTimeoutLayer = 1u << 7;  // a wait of the persistent decode layer ran out
constexpr uint32_t kStatusTimeoutMask =
    kStatusTimeoutGateUp | kStatusTimeoutDown | kStatusTimeoutRouter | kStatusTimeoutCheck |
    kStatusTimeoutLayer;

// A bounded pipeline wait gives up after this long (the longest legitimate
// wait is one tile's mainloop, well under a millisecond).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

// ---------------------------------------------------------- workspace --

struct Layout {
  size_t status, route_part, router_w, blk_counts, blk_base, plan, x_perm, h, out_perm;
  size_t cap_counts, cap_offsets, cap_perm, cap_inv, cap_wperm;  // dropless dispatch under a capacity
  size_t split_part;
  size_t logits, topk_ids, topk_w, gap, counts, offsets, perm_src, inv_pos, w_perm;
  size_t total;
  int route_splits;
  int nblk;      // dispatch blocks
  int nseg;      // E (+1 with the shared expert)
  int64_t rows;  // R = T*k (+T)
};

// Host: workspace layout of a (validated) descriptor.
Layout make_layout(const moe_layer_desc_t &d);
// K splits of the tensor-core router for `nsm` SMs (monotone in nsm); the
// workspace is sized for kRouteSizingSms, launches use min(SMs, that).
int route_splits(int T, int E, int H, int nsm);
constexpr int kRouteSizingSms = 256;

// Tile plan layout inside the plan buffer (int32):
//   [0, nseg]                 segment row offsets (nseg+1)
//   [nseg+1, 2nseg+1]         gate/up tile prefix (nseg+1)
//   [2nseg+2, 3nseg+2]        down tile prefix (nseg+1)
//   [3nseg+3], [3nseg+4]      split-K factor S of the gate/up and down GEMM
inline int plan_ints(int nseg) { return 3 * (nseg + 1) + 4; }

// Split-K for small batches: when every tile has at most kSplitMaxRows token
// rows and there are too few tiles to occupy the GPU, each tile's K range is
// cut into S pieces (S <= kMaxSplit, at most kMaxSplitTiles pieces in all);
// each piece writes an fp32 partial [NA][kBM][kSplitMaxRows] (NA = 2 for
// gate/up, 1 for down) and the last to
// finish adds them in split order.
constexpr int kSplitMaxRows = 32;
constexpr int kMaxSplit = 16;
constexpr int kMaxSplitTiles = 1024;

// Persistent decode layer (decode_layer.cu): batches of up to kDecodeMaxT
// tokens run the whole layer in one cooperative launch of one CTA per SM.
// Its counters follow the split-K counters in the status block: the
// arrival counts of its two grid barriers (after the router; before the
// combine), a count of finished CTAs, one arrival counter per CTA and work
// region (gate/up, down) for the pieces of a tile split between CTAs, and
// one readiness counter per segment (gate/up tiles finished).  Each returns
// to zero by the end of the launch (the generation only ever grows).
constexpr int kDecodeMaxT = 16;
constexpr int kDecodeMaxCtas = 256;
// words: +0 first grid barrier's arrivals, +1 second's, +2 finished CTAs
constexpr int kDecodeBarrierWord = kSplitCounterWord + 2 * kMaxSplitTiles;
constexpr int kDecodePieceWord = kDecodeBarrierWord + 32;
constexpr int kDecodeSegWord = kDecodePieceWord + 2 * kDecodeMaxCtas;
constexpr size_t kStatusBlockBytes = (size_t)(kDecodeSegWord + kMaxE + 16) * 4;

// ------------------------------------------------------ argument checks --
// Host-side validation shared by every entry point (api.cu, noalloc.cu):
// descriptor enums and shape limits (MOE_ERR_INVALID_ARG /
// MOE_ERR_UNSUPPORTED_SHAPE), 16-byte aligned non-null pointers, and the
// current device's compute capability (10.3, cached per device).
moe_status_t validate_desc(const moe_layer_desc_t *d);
bool ok_ptr(const void *p);  // non-null and 16-byte aligned
bool ok_opt(const void *p);  // null, or 16-byte aligned
moe_status_t check_device();

// ------------------------------------------------------------- launches --
// Each returns cudaSuccess or the launch error.
cudaError_t launch_router_logits(const __nv_bfloat16 *x, const float *w_router, int T, int H, int E,
                                 int splits, __nv_bfloat16 *w_split, float *partial,
                                 uint32_t *status, cudaStream_t s);
cudaError_t launch_route_small(const __nv_bfloat16 *x, const float *w_router,
                               const float *sel_bias, int T, int H, int E, int k, int gating,
                               float *logits, int32_t *ids, float *w, float *gap,
                               uint32_t *counter, cudaStream_t s);
cudaError_t launch_topk_gating(const float *partial, int splits, const float *sel_bias, int T,
                               int E, int k, int gating, float *logits, int32_t *ids, float *w,
                               float *gap, cudaStream_t s);
// Where a dispatch kernel also writes the GEMMs' tile plan (plan != null).
struct PlanArgs {
  int32_t *plan;
  int T, k, H, I, shared, num_sms;
  uint32_t *status;
};
// plan may be null; otherwise the dispatch also writes the tile plan, so the
// expert GEMMs can read it before waiting on the gather kernel.
cudaError_t launch_dispatch(const int32_t *ids, const float *topk_w, int T, int k, int E,
                            int32_t *blk_counts, int32_t *blk_base, int32_t *counts,
                            int32_t *offsets, int32_t *perm_src, int32_t *inv_pos, float *w_perm,
                            uint32_t *status, int32_t *plan, int H, int I, int shared,
                            cudaStream_t s);
// inv_pos may be null: then one warp per x_perm row (the standalone FFN call,
// and layer forwards whose x is at most kGatherByTokenBytes).  plan may be
// null (the dispatch wrote it); otherwise one more block writes it.
// (measured: a 4 MB threshold made the Qwen3 T=1024 forward 5 us slower)
#ifndef MOE_GATHER_TOKEN_KB
#define MOE_GATHER_TOKEN_KB 8192
#endif
constexpr int64_t kGatherByTokenBytes = (int64_t)MOE_GATHER_TOKEN_KB << 10;
// h: the first 256 rows past the last segment (if the segments end before
// T*k) are zeroed.
// to_fp16: x_perm rows in fp16 (the token operand of the FP8-weight GEMMs)
cudaError_t launch_gather_plan(const __nv_bfloat16 *x, const int32_t *perm_src,
                               const int32_t *inv_pos, const int32_t *offsets, int T, int k, int E,
                               int H, int I, int shared, __nv_bfloat16 *x_perm, __nv_bfloat16 *h,
                               int32_t *plan, uint32_t *status, cudaStream_t s,
                               bool to_fp16 = false);
// split_part: kMaxSplitTiles x 2 x kBM x kSplitMaxRows fp32; split_cnt: the
// GEMM's kMaxSplitTiles arrival counters (in the workspace status block).
// plan_early: the plan was written before the kernel preceding the GEMM
// (by the dispatch), so the GEMM may read it before waiting on that kernel.
// pair_ok: prefill-sized batches may run on CTA pairs (gemm_pair_supported)
cudaError_t launch_expert_gateup(const moe_layer_desc_t &d, const void *w13, const void *w13_shared,
                                 const __nv_bfloat16 *x_perm, const int32_t *plan, int plan_early,
                                 float *split_part, uint32_t *split_cnt, __nv_bfloat16 *h,
                                 uint32_t *status, bool pair_ok, cudaStream_t s);
cudaError_t launch_expert_down(const moe_layer_desc_t &d, const void *w2, const void *w2_shared,
                               const __nv_bfloat16 *h, const int32_t *plan, const float *w_perm,
                               float *split_part, uint32_t *split_cnt, __half *out_perm,
                               uint32_t *status, bool pair_ok, cudaStream_t s);

// Token-row tensor maps with box heights 16, 32, ..., 256 rows (x kStageKB K
// blocks).
struct TokenMaps {
  CUtensorMap m[16];
};
// The expert GEMMs with FP8 (E4M3) weights and per-128x128-block exponents
// (w_scale, as moe_layer_weights_fp8_t lays them out) for the kernel chain:
// act = fp16 token rows [R][K] (x_perm or h), out = fp16 h or out_perm.
cudaError_t launch_expert_gemm_fp8(bool gate_up, const moe_layer_desc_t &d, const void *w,
                                   const int8_t *w_scale, const void *w_sh,
                                   const int8_t *w_sh_scale, const void *act,
                                   const int32_t *plan, const float *w_perm, void *out,
                                   uint32_t *status, cudaStream_t s);
// The expert GEMMs on CTA pairs (tcgen05.mma.cta_group::2): shapes it takes
// (K a whole number of stages, output columns a whole number of pair tiles,
// enough rows per expert: gate/up T*k >= 256*E, down 64*E when I >= 2048),
// and its launch.  a / a_sh: this CTA's weight rows (gate/up:
// 64 gate + 64 up rows; down: 128 W2 rows), kStageKB K blocks per box.
bool gemm_pair_supported(const moe_layer_desc_t &d, bool gate_up);
cudaError_t launch_expert_gemm_pair(bool gate_up, const CUtensorMap &a, const CUtensorMap &a_sh,
                                    const TokenMaps &b, const int32_t *plan, int nseg, int E,
                                    int K, int out_cols, int64_t Na, const float *w_perm,
                                    void *out, uint32_t *status, cudaStream_t s);
// shared_base: null (the shared expert's rows at T*k) or a device pointer to
// their first row (offsets[E] under a capacity limit).
cudaError_t launch_combine(const __half *out_perm, const int32_t *inv_pos,
                           const float *topk_w, int T, int k, int H, int shared, __nv_bfloat16 *y,
                           cudaStream_t s, const int32_t *shared_base = nullptr);
// Capacity limit (dispatch.cu): from a dropless dispatch (counts, offsets,
// perm_src, w_perm of T*k assignments) the layout of the kept assignments --
// the first C of each expert in token order -- with inv_pos = -1 for a
// dropped assignment and perm_src = -1 past the kept rows.
cudaError_t launch_capacity(const int32_t *counts, const int32_t *offsets, const int32_t *perm_src,
                            const float *w_perm, int T, int k, int E, int C, int32_t *counts_c,
                            int32_t *offsets_c, int32_t *perm_c, int32_t *inv_c, float *w_perm_c,
                            cudaStream_t s);
// The persistent decode layer (decode_layer.cu): the whole forward in one
// cooperative launch for shapes decode_layer_supported accepts.
bool decode_layer_supported(const moe_layer_desc_t &d);
cudaError_t launch_decode_layer(const moe_layer_desc_t &d, const moe_layer_weights_t &w,
                                const __nv_bfloat16 *x, __nv_bfloat16 *y, void *workspace,
                                const Layout &L, cudaStream_t s);
// Two CTAs of one cooperative launch meet at the decode layer's grid barrier
// sized for three: both waits run out after kWaitLimitNs and latch
// kStatusTimeoutLayer (decode_layer.cu).
cudaError_t launch_grid_wait_check(uint32_t *status_block, cudaStream_t s);
// Tensor maps of the expert GEMMs (expert_gemm.cu): weights [E][P][rows][K]
// as {64, rows, P, K/64, E} with boxes of box_rows rows and kStageKB K
// blocks; token rows [R][K] as {64, R, K/64} with boxes of box_rows rows.
bool weight_map(CUtensorMap *m, const void *w, int K, int rows, int P, int E, int box_rows);
bool act_map(CUtensorMap *m, const void *a, int K, int64_t R, int box_rows,
             int kblocks = kStageKB);
// The same weight view over E4M3 codes (one byte each), unswizzled boxes.
bool weight_map_u8(CUtensorMap *m, const void *w, int K, int rows, int P, int E, int box_rows);
// FP8 expert weights (quantize.cu, decode_layer.cu).
cudaError_t launch_quantize_fp8(const __nv_bfloat16 *w, int n, int rows, int K, uint8_t *q,
                                int8_t *scale, cudaStream_t s);
cudaError_t launch_decode_layer_fp8(const moe_layer_desc_t &d, const moe_layer_weights_fp8_t &w,
                                    const __nv_bfloat16 *x, __nv_bfloat16 *y, void *workspace,
                                    const Layout &L, cudaStream_t s);
// One thread waits on an mbarrier nothing arrives on (waitcheck.cu).
cudaError_t launch_bounded_wait_check(uint32_t *status, cudaStream_t s);
// EP <-> TP expert-weight reshard permute (reshard.cu); a null source skips
// that tensor.  unpack = 0: EP layout -> per-peer chunks; 1: the inverse.
cudaError_t launch_reshard(int E_local, int H, int I, int P, const void *w13_src, void *w13_dst,
                           const void *w2_src, void *w2_dst, int unpack, cudaStream_t st);

int num_sms();  // of the current device (cached)

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first,
// strides in bytes for dims 1..rank-1.  False if the encoder is unavailable
// or rejects the arguments.
bool encode_bf16_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                     const cuuint64_t *strides, const cuuint32_t *box);

// ----------------------------------------------------- device helpers --

// Programmatic dependent launch.  Every kernel of the path is launched with
// programmatic stream serialization, so its launch and its input-independent
// prologue (barrier set-up, TMEM allocation, descriptor prefetch) overlap the
// previous kernel's tail.  Each kernel calls pdl_wait() before it reads
// memory that an earlier stream operation wrote, then
// pdl_launch_dependents() so that the next kernel may launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Two floats to one word of two 16-bit values (lo in bits 0-15), rounded to
// nearest even: bf16, or fp16 with magnitudes past 65504 saturated to it.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t pack_f16x2_satfinite(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// max(a, b) that returns NaN when either is NaN
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// --- mbarrier ---
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Gives up (returns false) when the
// CTA's abort flag is raised or after kWaitLimitNs; on its own timeout it
// raises the abort flag and latches `code` in the global status word.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *status, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  *abort_flag = 1;
  atomicOr(status, code);
  return false;
}

// Short bounded wait used only while draining after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs / 10) return false;
  }
  return false;
}

// Acquire load of a flag another CTA releases (gpu scope).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders this thread's generic-proxy global accesses with its async-proxy
// (TMA) accesses: written by a generic store, read by a tensor copy.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bulk copy of `bytes` (a multiple of 16) from global to shared memory, both
// addresses 16-byte aligned; completion on an mbarrier.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses with later
// async-proxy (bulk / tensor copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --- TMA (tensor tiles, global -> shared, completion on an mbarrier) ---
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0,
                                            int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// --- tcgen05: tensor memory, MMA, loads ---
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 op this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns; thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 64 bf16 (128 B), 8-row core groups 1024 B
// apart.  Fields: start address >> 4 (bits 0-13), leading byte offset >> 4
// (bits 16-29, unused for this layout), stride byte offset >> 4 (bits
// 32-45), descriptor version 1 (bits 46-47), swizzle mode 2 = 128 B (bits
// 61-63).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

}  // namespace moe
