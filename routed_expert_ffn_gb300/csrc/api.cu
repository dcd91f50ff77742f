// C ABI of the MoE FFN layer forward: argument validation, workspace layout,
// the stage calls and the fused layer forward.  Declarations and the meaning
// of every argument are in include/moe.h.
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

Layout make_layout(const moe_layer_desc_t &d) {
  Layout L;
  memset(&L, 0, sizeof L);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 1024);
    return o;
  };
  const int64_t Na = (int64_t)d.T * d.k;
  const int shared = d.has_shared_expert ? 1 : 0;
  L.rows = Na + (shared ? d.T : 0);
  L.nseg = d.E + shared;
  L.route_splits = route_splits(d.T, d.E, d.H, kRouteSizingSms);  // the most a launch uses
  const int64_t chunk = dispatch_chunk(Na);
  L.nblk = (int)((Na + chunk - 1) / chunk);
  L.status = take(kStatusBlockBytes);
  L.route_part = take((size_t)L.route_splits * d.T * d.E * 4);
  L.router_w = take((size_t)3 * d.E * d.H * 2);
  L.blk_counts = take((size_t)L.nblk * d.E * 4);
  L.blk_base = take((size_t)L.nblk * d.E * 4);
  L.plan = take((size_t)plan_ints(L.nseg) * 4);
  L.split_part = take((size_t)kMaxSplitTiles * 2 * kBM * kSplitMaxRows * 4);
  L.logits = take((size_t)d.T * d.E * 4);
  L.topk_ids = take((size_t)Na * 4);
  L.topk_w = take((size_t)Na * 4);
  L.gap = take((size_t)d.T * 4);
  L.counts = take((size_t)d.E * 4);
  L.offsets = take((size_t)(d.E + 1) * 4);
  L.perm_src = take((size_t)Na * 4);
  L.inv_pos = take((size_t)Na * 4);
  L.w_perm = take((size_t)Na * 4);
  L.cap_counts = take((size_t)d.E * 4);
  L.cap_offsets = take((size_t)(d.E + 1) * 4);
  L.cap_perm = take((size_t)Na * 4);
  L.cap_inv = take((size_t)Na * 4);
  L.cap_wperm = take((size_t)Na * 4);
  L.x_perm = take((size_t)L.rows * d.H * 2);
  L.h = take((size_t)L.rows * d.I * 2);
  L.out_perm = take((size_t)L.rows * d.H * 2);
  L.total = off;
  return L;
}

moe_status_t validate_desc(const moe_layer_desc_t *d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->gating < MOE_GATE_TOPK_SOFTMAX || d->gating > MOE_GATE_SIGMOID_BIAS_RENORM)
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared_expert != 0 && d->has_shared_expert != 1) return MOE_ERR_INVALID_ARG;
  if (d->T < 1 || d->T > kMaxT) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->E < 1 || d->E > kMaxE) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->k < 1 || d->k > d->E || d->k > kMaxK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)d->T * d->k > kMaxAssign) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->H < 64 || d->H > 16384 || d->H % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d->I < 64 || d->I > 32768 || d->I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

bool ok_ptr(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_opt(const void *p) { return p == nullptr || ok_ptr(p); }

moe_status_t check_device() {
  static int8_t state[64] = {};  // 0 unknown, 1 supported, -1 not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (state[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    state[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return state[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

}  // namespace moe

using namespace moe;

namespace {

// Common prologue of the compute calls: descriptor and workspace (host only;
// the device check comes after every argument has been validated).
moe_status_t prologue(const moe_layer_desc_t *d, void *ws, size_t ws_bytes, Layout *L) {
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (ws != nullptr) {
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    *L = make_layout(*d);
    if (ws_bytes < L->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  }
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

const __nv_bfloat16 *bf(const void *p) { return static_cast<const __nv_bfloat16 *>(p); }

// Router + gating: one fused launch for small batches, else the tensor-core
// router (split-K partials) followed by the gating kernel.
cudaError_t route(const moe_layer_desc_t &d, const Layout &L, const __nv_bfloat16 *x,
                  const float *w_router, const float *sel_bias, float *logits, int32_t *ids,
                  float *w, float *gap, void *workspace, cudaStream_t s) {
  uint32_t *status = at<uint32_t>(workspace, L.status);
  if (d.T <= kSmallRouteT)
    return launch_route_small(x, w_router, sel_bias, d.T, d.H, d.E, d.k, d.gating, logits, ids, w,
                              gap, status + kRouteCounterWord, s);
  float *part = at<float>(workspace, L.route_part);
  const int splits = route_splits(d.T, d.E, d.H, std::min(num_sms(), kRouteSizingSms));
  cudaError_t e = launch_router_logits(x, w_router, d.T, d.H, d.E, splits,
                                       at<__nv_bfloat16>(workspace, L.router_w), part, status, s);
  if (e == cudaSuccess)
    e = launch_topk_gating(part, splits, sel_bias, d.T, d.E, d.k, d.gating, logits, ids, w, gap, s);
  return e;
}
__nv_bfloat16 *bfw(void *p) { return static_cast<__nv_bfloat16 *>(p); }

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_layer_desc_t *d) {
  if (validate_desc(d) != MOE_OK) return 0;
  return make_layout(*d).total;
}

moe_status_t moe_workspace_layout(const moe_layer_desc_t *d, moe_workspace_layout_t *out) {
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(*d);
  out->status = L.status;
  out->logits = L.logits;
  out->topk_ids = L.topk_ids;
  out->topk_w = L.topk_w;
  out->gap = L.gap;
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->perm_src = L.perm_src;
  out->inv_pos = L.inv_pos;
  out->w_perm = L.w_perm;
  out->x_perm = L.x_perm;
  out->h = L.h;
  out->out_perm = L.out_perm;
  out->plan = L.plan;
  out->total = L.total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void *workspace, size_t ws_bytes, moe_stream_t stream) {
  if (workspace == nullptr || ws_bytes < kStatusBlockBytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, kStatusBlockBytes, (cudaStream_t)stream));
}

moe_status_t moe_get_device_status(void *workspace, size_t ws_bytes, moe_stream_t stream,
                                   int32_t clear, int32_t *raw) {
  if (workspace == nullptr || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (clear) {
    if (cudaMemsetAsync(workspace, 0, sizeof word, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (raw != nullptr) *raw = (int32_t)word;
  if (word & kStatusTimeoutMask) return MOE_ERR_TIMEOUT;
  if (word & (kStatusBadExpertId | kStatusBadOffsets | kStatusRange)) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}

moe_status_t moe_check_bounded_wait(void *workspace, size_t ws_bytes, moe_stream_t stream) {
  if (workspace == nullptr || ws_bytes < kStatusBlockBytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return cuda_status(
      launch_bounded_wait_check(static_cast<uint32_t *>(workspace), (cudaStream_t)stream));
}

const char *moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (NULL or misaligned pointer, bad enum)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "shape outside the supported limits";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than moe_workspace_size()";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_DEVICE_CHECK:
      return "device check failed (expert id or offsets out of range, or an expert output "
             "beyond the fp16 range of out_perm)";
    case MOE_ERR_TIMEOUT: return "a bounded device pipeline wait timed out";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3";
    default: return "unknown status";
  }
}

moe_status_t moe_route(const moe_layer_desc_t *d, const void *x, const float *w_router,
                       const float *sel_bias, float *logits, int32_t *topk_ids, float *topk_w,
                       float *boundary_gap, void *workspace, size_t ws_bytes,
                       moe_stream_t stream) {
  if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status_t st = prologue(d, workspace, ws_bytes, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(x) || !ok_ptr(w_router) || !ok_ptr(logits) || !ok_ptr(topk_ids) || !ok_ptr(topk_w) ||
      !ok_opt(boundary_gap))
    return MOE_ERR_INVALID_ARG;
  if (d->gating == MOE_GATE_SIGMOID_BIAS_RENORM && !ok_ptr(sel_bias)) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return cuda_status(route(*d, L, bf(x), w_router, sel_bias, logits, topk_ids, topk_w,
                           boundary_gap, workspace, (cudaStream_t)stream));
}

moe_status_t moe_build_dispatch(const moe_layer_desc_t *d, const int32_t *topk_ids,
                                const float *topk_w, int32_t *counts, int32_t *offsets,
                                int32_t *perm_src, int32_t *inv_pos, float *w_perm,
                                void *workspace, size_t ws_bytes, moe_stream_t stream) {
  if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status_t st = prologue(d, workspace, ws_bytes, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(topk_ids) || !ok_ptr(counts) || !ok_ptr(offsets) || !ok_ptr(perm_src) ||
      !ok_ptr(inv_pos) || !ok_opt(topk_w) || !ok_opt(w_perm))
    return MOE_ERR_INVALID_ARG;
  if (w_perm != nullptr && topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t e = launch_dispatch(topk_ids, topk_w, d->T, d->k, d->E,
                                  at<int32_t>(workspace, L.blk_counts),
                                  at<int32_t>(workspace, L.blk_base), counts, offsets, perm_src,
                                  inv_pos, w_perm, at<uint32_t>(workspace, L.status), nullptr,
                                  d->H, d->I, d->has_shared_expert, (cudaStream_t)stream);
  return cuda_status(e);
}

moe_status_t moe_grouped_swiglu_ffn(const moe_layer_desc_t *d, const void *x,
                                    const int32_t *perm_src, const int32_t *offsets,
                                    const float *w_perm, const void *w13, const void *w2,
                                    const void *w13_shared, const void *w2_shared,
                                    void *out_perm, void *workspace, size_t ws_bytes,
                                    moe_stream_t stream) {
  if (workspace == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status_t st = prologue(d, workspace, ws_bytes, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(x) || !ok_ptr(perm_src) || !ok_ptr(offsets) || !ok_opt(w_perm) || !ok_ptr(w13) ||
      !ok_ptr(w2) || !ok_ptr(out_perm))
    return MOE_ERR_INVALID_ARG;
  if (d->has_shared_expert && (!ok_ptr(w13_shared) || !ok_ptr(w2_shared)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t *status = at<uint32_t>(workspace, L.status);
  int32_t *plan = at<int32_t>(workspace, L.plan);
  __nv_bfloat16 *x_perm = at<__nv_bfloat16>(workspace, L.x_perm);
  __nv_bfloat16 *h = at<__nv_bfloat16>(workspace, L.h);
  float *split_part = at<float>(workspace, L.split_part);
  uint32_t *split_cnt = at<uint32_t>(workspace, L.status) + kSplitCounterWord;
  cudaError_t e = launch_gather_plan(bf(x), perm_src, nullptr, offsets, d->T, d->k, d->E, d->H,
                                     d->I, d->has_shared_expert, x_perm, h, plan, status, s);
  if (e == cudaSuccess)
    e = launch_expert_gateup(*d, w13, w13_shared, x_perm, plan, 0, split_part, split_cnt, h,
                             status, true, s);
  if (e == cudaSuccess)
    e = launch_expert_down(*d, w2, w2_shared, h, plan, w_perm, split_part,
                           split_cnt + kMaxSplitTiles, static_cast<__half *>(out_perm), status, true, s);
  return cuda_status(e);
}

moe_status_t moe_combine(const moe_layer_desc_t *d, const void *out_perm, const int32_t *inv_pos,
                         const float *topk_w, void *y, moe_stream_t stream) {
  Layout L;
  moe_status_t st = prologue(d, nullptr, 0, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(out_perm) || !ok_ptr(inv_pos) || !ok_opt(topk_w) || !ok_ptr(y))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  return cuda_status(launch_combine(static_cast<const __half *>(out_perm), inv_pos, topk_w, d->T,
                                    d->k, d->H,
                                    d->has_shared_expert, bfw(y), (cudaStream_t)stream));
}

moe_status_t moe_layer_forward_ex(const moe_layer_desc_t *d, const moe_layer_weights_t *w,
                                  const void *x, void *y, void *workspace, size_t ws_bytes,
                                  moe_stream_t stream, moe_event_t const *stage_events,
                                  int32_t path) {
  if (workspace == nullptr || w == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status_t st = prologue(d, workspace, ws_bytes, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(x) || !ok_ptr(y) || !ok_ptr(w->w_router) || !ok_ptr(w->w13) || !ok_ptr(w->w2))
    return MOE_ERR_INVALID_ARG;
  if (d->gating == MOE_GATE_SIGMOID_BIAS_RENORM && !ok_ptr(w->sel_bias)) return MOE_ERR_INVALID_ARG;
  if (d->has_shared_expert && (!ok_ptr(w->w13_shared) || !ok_ptr(w->w2_shared)))
    return MOE_ERR_INVALID_ARG;
  if (path < MOE_PATH_AUTO || path > MOE_PATH_CHAIN_ONE_SM) return MOE_ERR_INVALID_ARG;
  // the expert GEMMs may take CTA-pair tiles (prefill batches) unless the
  // one-SM chain is asked for
  const bool pair_ok = path != MOE_PATH_CHAIN_ONE_SM;
  const bool persistent_ok = decode_layer_supported(*d);
  if (path == MOE_PATH_PERSISTENT && !persistent_ok) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  auto mark = [&](int i) -> cudaError_t {
    return stage_events ? cudaEventRecord((cudaEvent_t)stage_events[i], s) : cudaSuccess;
  };
  if (path == MOE_PATH_PERSISTENT || (path == MOE_PATH_AUTO && persistent_ok)) {
    // the whole layer in one launch: every stage boundary is at its end
    cudaError_t e = mark(0);
    if (e == cudaSuccess)
      e = launch_decode_layer(*d, *w, bf(x), bfw(y), workspace, L, s);
    for (int i = 1; e == cudaSuccess && i < MOE_STAGE_EVENTS; ++i) e = mark(i);
    return cuda_status(e);
  }
  uint32_t *status = at<uint32_t>(workspace, L.status);
  float *logits = at<float>(workspace, L.logits);
  int32_t *ids = at<int32_t>(workspace, L.topk_ids);
  float *tw = at<float>(workspace, L.topk_w);
  int32_t *offsets = at<int32_t>(workspace, L.offsets);
  int32_t *perm_src = at<int32_t>(workspace, L.perm_src);
  int32_t *inv_pos = at<int32_t>(workspace, L.inv_pos);
  float *w_perm = at<float>(workspace, L.w_perm);
  int32_t *plan = at<int32_t>(workspace, L.plan);
  __nv_bfloat16 *x_perm = at<__nv_bfloat16>(workspace, L.x_perm);
  __nv_bfloat16 *h = at<__nv_bfloat16>(workspace, L.h);
  __half *out_perm = at<__half>(workspace, L.out_perm);
  float *split_part = at<float>(workspace, L.split_part);
  uint32_t *split_cnt = at<uint32_t>(workspace, L.status) + kSplitCounterWord;
  cudaError_t e = mark(0);
  if (e == cudaSuccess)
    e = route(*d, L, bf(x), w->w_router, w->sel_bias, logits, ids, tw, at<float>(workspace, L.gap),
              workspace, s);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess)
    e = launch_dispatch(ids, tw, d->T, d->k, d->E, at<int32_t>(workspace, L.blk_counts),
                        at<int32_t>(workspace, L.blk_base), at<int32_t>(workspace, L.counts),
                        offsets, perm_src, inv_pos, w_perm, status, plan, d->H, d->I,
                        d->has_shared_expert, s);
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess)
    // token-order gather (x read once) once x is too large to stay in L2
    // between its k reads; row order keeps more warps busy for small batches
    e = launch_gather_plan(bf(x), perm_src,
                           (int64_t)d->T * d->H * 2 > kGatherByTokenBytes ? inv_pos : nullptr,
                           offsets, d->T, d->k, d->E, d->H, d->I, d->has_shared_expert, x_perm,
                           h, nullptr, status, s);  // the dispatch wrote the plan
  if (e == cudaSuccess) e = mark(3);
  if (e == cudaSuccess)
    e = launch_expert_gateup(*d, w->w13, w->w13_shared, x_perm, plan, 1, split_part, split_cnt, h,
                             status, pair_ok, s);
  if (e == cudaSuccess) e = mark(4);
  if (e == cudaSuccess)
    e = launch_expert_down(*d, w->w2, w->w2_shared, h, plan, w_perm, split_part,
                           split_cnt + kMaxSplitTiles, out_perm, status, pair_ok, s);
  if (e == cudaSuccess) e = mark(5);
  if (e == cudaSuccess)
    e = launch_combine(out_perm, inv_pos, nullptr, d->T, d->k, d->H, d->has_shared_expert, bfw(y), s);
  if (e == cudaSuccess) e = mark(6);
  return cuda_status(e);
}

moe_status_t moe_layer_forward(const moe_layer_desc_t *d, const moe_layer_weights_t *w,
                               const void *x, void *y, void *workspace, size_t ws_bytes,
                               moe_stream_t stream, moe_event_t const *stage_events) {
  return moe_layer_forward_ex(d, w, x, y, workspace, ws_bytes, stream, stage_events,
                              MOE_PATH_AUTO);
}

int32_t moe_expert_capacity(int64_t cf_num, int64_t cf_den, int32_t T, int32_t k, int32_t E) {
  if (cf_num <= 0 || cf_den <= 0 || T < 1 || k < 1 || E < 1) return 0;
  if (cf_num > ((int64_t)1 << 30) || cf_den > ((int64_t)1 << 30)) return 0;
  const int64_t num = cf_num * ((int64_t)T * k), den = cf_den * E;  // < 2^55, < 2^40
  const int64_t c = (num + den - 1) / den;
  return c > ((int64_t)1 << 30) ? ((int32_t)1 << 30) : (int32_t)c;
}

moe_status_t moe_layer_forward_capacity(const moe_layer_desc_t *d, const moe_layer_weights_t *w,
                                        const void *x, void *y, int32_t capacity,
                                        void *workspace, size_t ws_bytes, moe_stream_t stream) {
  if (workspace == nullptr || w == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status_t st = prologue(d, workspace, ws_bytes, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(x) || !ok_ptr(y) || !ok_ptr(w->w_router) || !ok_ptr(w->w13) || !ok_ptr(w->w2))
    return MOE_ERR_INVALID_ARG;
  if (d->gating == MOE_GATE_SIGMOID_BIAS_RENORM && !ok_ptr(w->sel_bias)) return MOE_ERR_INVALID_ARG;
  if (d->has_shared_expert && (!ok_ptr(w->w13_shared) || !ok_ptr(w->w2_shared)))
    return MOE_ERR_INVALID_ARG;
  if (capacity < 1) return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t *status = at<uint32_t>(workspace, L.status);
  float *tw = at<float>(workspace, L.topk_w);
  int32_t *ids = at<int32_t>(workspace, L.topk_ids);
  int32_t *offsets = at<int32_t>(workspace, L.offsets);
  int32_t *perm_src = at<int32_t>(workspace, L.perm_src);
  int32_t *inv_pos = at<int32_t>(workspace, L.inv_pos);
  float *w_perm = at<float>(workspace, L.w_perm);
  int32_t *plan = at<int32_t>(workspace, L.plan);
  __nv_bfloat16 *x_perm = at<__nv_bfloat16>(workspace, L.x_perm);
  __nv_bfloat16 *h = at<__nv_bfloat16>(workspace, L.h);
  __half *out_perm = at<__half>(workspace, L.out_perm);
  float *split_part = at<float>(workspace, L.split_part);
  uint32_t *split_cnt = at<uint32_t>(workspace, L.status) + kSplitCounterWord;
  // route; the dropless dispatch into scratch; the kept assignments' layout
  // into the workspace's routing buffers; then the chain as without a limit,
  // the tile plan written by the gather from the kept layout
  cudaError_t e = route(*d, L, bf(x), w->w_router, w->sel_bias, at<float>(workspace, L.logits),
                        ids, tw, at<float>(workspace, L.gap), workspace, s);
  if (e == cudaSuccess)
    e = launch_dispatch(ids, tw, d->T, d->k, d->E, at<int32_t>(workspace, L.blk_counts),
                        at<int32_t>(workspace, L.blk_base), at<int32_t>(workspace, L.cap_counts),
                        at<int32_t>(workspace, L.cap_offsets), at<int32_t>(workspace, L.cap_perm),
                        at<int32_t>(workspace, L.cap_inv), at<float>(workspace, L.cap_wperm),
                        status, nullptr, d->H, d->I, d->has_shared_expert, s);
  if (e == cudaSuccess)
    e = launch_capacity(at<int32_t>(workspace, L.cap_counts), at<int32_t>(workspace, L.cap_offsets),
                        at<int32_t>(workspace, L.cap_perm), at<float>(workspace, L.cap_wperm),
                        d->T, d->k, d->E, capacity, at<int32_t>(workspace, L.counts), offsets,
                        perm_src, inv_pos, w_perm, s);
  if (e == cudaSuccess)
    e = launch_gather_plan(bf(x), perm_src,
                           (int64_t)d->T * d->H * 2 > kGatherByTokenBytes ? inv_pos : nullptr,
                           offsets, d->T, d->k, d->E, d->H, d->I, d->has_shared_expert, x_perm,
                           h, plan, status, s);
  if (e == cudaSuccess)
    e = launch_expert_gateup(*d, w->w13, w->w13_shared, x_perm, plan, 0, split_part, split_cnt, h,
                             status, true, s);
  if (e == cudaSuccess)
    e = launch_expert_down(*d, w->w2, w->w2_shared, h, plan, w_perm, split_part,
                           split_cnt + kMaxSplitTiles, out_perm, status, true, s);
  if (e == cudaSuccess)
    e = launch_combine(out_perm, inv_pos, nullptr, d->T, d->k, d->H, d->has_shared_expert, bfw(y),
                       s, offsets + d->E);
  return cuda_status(e);
}

moe_status_t moe_quantize_fp8(const void *w, int32_t n, int32_t rows, int32_t K, void *q,
                              int8_t *scale_exp, moe_stream_t stream) {
  if (!ok_ptr(w) || !ok_ptr(q) || scale_exp == nullptr) return MOE_ERR_INVALID_ARG;
  if (n < 1 || rows < 1 || K < 64 || K % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)n * rows * K >= ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return cuda_status(launch_quantize_fp8(bf(w), n, rows, K, static_cast<uint8_t *>(q), scale_exp,
                                         (cudaStream_t)stream));
}

moe_status_t moe_layer_forward_fp8(const moe_layer_desc_t *d, const moe_layer_weights_fp8_t *w,
                                   const void *x, void *y, void *workspace, size_t ws_bytes,
                                   moe_stream_t stream) {
  if (workspace == nullptr || w == nullptr) return MOE_ERR_INVALID_ARG;
  Layout L;
  moe_status_t st = prologue(d, workspace, ws_bytes, &L);
  if (st != MOE_OK) return st;
  if (!ok_ptr(x) || !ok_ptr(y) || !ok_ptr(w->w_router) || !ok_ptr(w->w13) || !ok_ptr(w->w2) ||
      w->w13_scale == nullptr || w->w2_scale == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (d->gating == MOE_GATE_SIGMOID_BIAS_RENORM && !ok_ptr(w->sel_bias)) return MOE_ERR_INVALID_ARG;
  if (d->has_shared_expert && (!ok_ptr(w->w13_shared) || !ok_ptr(w->w2_shared) ||
                               w->w13_shared_scale == nullptr || w->w2_shared_scale == nullptr))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (decode_layer_supported(*d))
    return cuda_status(launch_decode_layer_fp8(*d, *w, bf(x), bfw(y), workspace, L, s));
  // larger batches: the kernel chain with FP8 GEMMs on fp16 token rows
  uint32_t *status = at<uint32_t>(workspace, L.status);
  int32_t *ids = at<int32_t>(workspace, L.topk_ids);
  float *tw = at<float>(workspace, L.topk_w);
  int32_t *offsets = at<int32_t>(workspace, L.offsets);
  int32_t *perm_src = at<int32_t>(workspace, L.perm_src);
  int32_t *inv_pos = at<int32_t>(workspace, L.inv_pos);
  float *w_perm = at<float>(workspace, L.w_perm);
  int32_t *plan = at<int32_t>(workspace, L.plan);
  __nv_bfloat16 *x_perm = at<__nv_bfloat16>(workspace, L.x_perm);  // fp16 rows in this mode
  __nv_bfloat16 *h = at<__nv_bfloat16>(workspace, L.h);            // fp16 rows in this mode
  __half *out_perm = at<__half>(workspace, L.out_perm);
  cudaError_t e = route(*d, L, bf(x), w->w_router, w->sel_bias, at<float>(workspace, L.logits), ids,
                        tw, at<float>(workspace, L.gap), workspace, s);
  if (e == cudaSuccess)
    e = launch_dispatch(ids, tw, d->T, d->k, d->E, at<int32_t>(workspace, L.blk_counts),
                        at<int32_t>(workspace, L.blk_base), at<int32_t>(workspace, L.counts),
                        offsets, perm_src, inv_pos, w_perm, status, plan, d->H, d->I,
                        d->has_shared_expert, s);
  if (e == cudaSuccess)
    e = launch_gather_plan(bf(x), perm_src,
                           (int64_t)d->T * d->H * 2 > kGatherByTokenBytes ? inv_pos : nullptr,
                           offsets, d->T, d->k, d->E, d->H, d->I, d->has_shared_expert, x_perm, h,
                           nullptr, status, s, /*to_fp16=*/true);
  if (e == cudaSuccess)
    e = launch_expert_gemm_fp8(true, *d, w->w13, w->w13_scale, w->w13_shared, w->w13_shared_scale,
                               x_perm, plan, nullptr, h, status, s);
  if (e == cudaSuccess)
    e = launch_expert_gemm_fp8(false, *d, w->w2, w->w2_scale, w->w2_shared, w->w2_shared_scale, h,
                               plan, w_perm, out_perm, status, s);
  if (e == cudaSuccess)
    e = launch_combine(out_perm, inv_pos, nullptr, d->T, d->k, d->H, d->has_shared_expert, bfw(y), s);
  return cuda_status(e);
}

moe_status_t moe_check_bounded_grid_wait(void *workspace, size_t ws_bytes, moe_stream_t stream) {
  if (workspace == nullptr || ws_bytes < kStatusBlockBytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_ERR_INVALID_ARG;
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  return cuda_status(
      launch_grid_wait_check(static_cast<uint32_t *>(workspace), (cudaStream_t)stream));
}

// Shared checks of the two reshard calls (the two directions take the same
// shapes; src/dst are the inputs/outputs of the call).
static moe_status_t reshard_checks(int32_t E_local, int32_t H, int32_t I, int32_t P,
                                   const void *src13, const void *src2, const void *dst13,
                                   const void *dst2) {
  if ((src13 == nullptr) != (dst13 == nullptr) || (src2 == nullptr) != (dst2 == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (src13 == nullptr && src2 == nullptr) return MOE_ERR_INVALID_ARG;
  if (!ok_opt(src13) || !ok_opt(src2) || !ok_opt(dst13) || !ok_opt(dst2))
    return MOE_ERR_INVALID_ARG;
  if (E_local < 1 || H < 8 || I < 8 || P < 1 || H % 8 != 0 || I % P != 0 || (I / P) % 8 != 0)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const int64_t bytes = (int64_t)E_local * 2 * I * H * 2;  // W13; W2 is half of it
  if (bytes >= (int64_t)1 << 35) return MOE_ERR_UNSUPPORTED_SHAPE;
  auto overlap = [](const void *a, int64_t na, const void *b, int64_t nb) {
    if (a == nullptr || b == nullptr) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
  };
  const int64_t b13 = bytes, b2 = bytes / 2;
  if (overlap(src13, b13, dst13, b13) || overlap(src13, b13, dst2, b2) ||
      overlap(src2, b2, dst13, b13) || overlap(src2, b2, dst2, b2) ||
      overlap(dst13, b13, dst2, b2))
    return MOE_ERR_INVALID_ARG;
  return check_device();
}

moe_status_t moe_reshard_ep_to_tp_pack(int32_t E_local, int32_t H, int32_t I, int32_t P,
                                       const void *w13, const void *w2, void *w13_chunks,
                                       void *w2_chunks, moe_stream_t stream) {
  moe_status_t st = reshard_checks(E_local, H, I, P, w13, w2, w13_chunks, w2_chunks);
  if (st != MOE_OK) return st;
  return cuda_status(launch_reshard(E_local, H, I, P, w13, w13_chunks, w2, w2_chunks, 0,
                                   (cudaStream_t)stream));
}

moe_status_t moe_reshard_tp_to_ep_unpack(int32_t E_local, int32_t H, int32_t I, int32_t P,
                                         const void *w13_chunks, const void *w2_chunks,
                                         void *w13, void *w2, moe_stream_t stream) {
  moe_status_t st = reshard_checks(E_local, H, I, P, w13_chunks, w2_chunks, w13, w2);
  if (st != MOE_OK) return st;
  return cuda_status(launch_reshard(E_local, H, I, P, w13_chunks, w13, w2_chunks, w2, 1,
                                   (cudaStream_t)stream));
}

}  // extern "C"
