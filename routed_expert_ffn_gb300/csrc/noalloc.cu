// moe_build_dispatch_noalloc: the count / prefix-sum / permute dispatch for
// callers that cannot allocate device memory.
//
// Some callers have no way to obtain a scratch buffer: a plugin running inside
// a host framework that owns the whole device-memory budget and hands its
// extensions no allocator, or a latency-critical path that must not call
// cudaMalloc because the call can synchronise the device.  This entry point
// needs only its inputs and outputs: the dispatch's scratch (the per-block
// expert histograms and their prefix bases, plus one status word) lives in a
// fixed-size array in this library's device memory.
//
// The array is shared by every call in the process and keeps the previous
// call's contents; every scratch entry the dispatch reads is written earlier
// in the same call, and the status word is cleared at the start of each call.
// Two calls whose work overlaps on the GPU (for example on two streams with
// no ordering between them) race on the array.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Maximum scratch: one status word (padded to 256 bytes) plus two int32
// tables of nblk x E entries each.
constexpr size_t kNoAllocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

// Device address of g_dispatch_scratch per device.  The array's name in host
// code is only a host-side stand-in, never a device address; the real address
// is looked up once per device, with that device current, on the first call.
void *g_scratch_addr[64] = {};
std::mutex g_scratch_mutex;

moe_status_t scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_build_dispatch_noalloc(const moe_layer_desc_t *d,
                                                   const int32_t *topk_ids, const float *topk_w,
                                                   int32_t *counts, int32_t *offsets,
                                                   int32_t *perm_src, int32_t *inv_pos,
                                                   float *w_perm, int32_t *device_status,
                                                   moe_stream_t stream) {
  // the same argument checks as moe_build_dispatch (api.cu)
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (!ok_ptr(topk_ids) || !ok_ptr(counts) || !ok_ptr(offsets) || !ok_ptr(perm_src) ||
      !ok_ptr(inv_pos) || !ok_opt(topk_w) || !ok_opt(w_perm) ||
      (device_status != nullptr && (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0))
    return MOE_ERR_INVALID_ARG;
  if (w_perm != nullptr && topk_w == nullptr) return MOE_ERR_INVALID_ARG;

  // The scratch this batch needs must fit the fixed array.
  const int64_t Na = (int64_t)d->T * d->k;
  const int64_t chunk = dispatch_chunk(Na);
  const int64_t nblk = (Na + chunk - 1) / chunk;
  const size_t table = (size_t)nblk * d->E * sizeof(int32_t);
  if (256 + 2 * table > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;

  if ((st = check_device()) != MOE_OK) return st;

  void *base = nullptr;
  st = scratch_address(&base);
  if (st != MOE_OK) return st;
  unsigned char *scratch = static_cast<unsigned char *>(base);
  uint32_t *status = reinterpret_cast<uint32_t *>(scratch);
  int32_t *blk_counts = reinterpret_cast<int32_t *>(scratch + 256);
  int32_t *blk_base = reinterpret_cast<int32_t *>(scratch + 256 + table);

  cudaStream_t s = (cudaStream_t)stream;
  // Only the status word must start at zero: both tables are fully written
  // before they are read within this call.
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = launch_dispatch(topk_ids, topk_w, d->T, d->k, d->E, blk_counts, blk_base, counts, offsets,
                        perm_src, inv_pos, w_perm, status, nullptr, d->H, d->I,
                        d->has_shared_expert, s);
  if (e == cudaSuccess && device_status != nullptr)
    e = cudaMemcpyAsync(device_status, status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
