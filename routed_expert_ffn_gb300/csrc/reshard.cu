// Local permute of an expert-weight reshard between expert parallelism (EP)
// and tensor parallelism (TP) (Moebius, section 3.1 "Weights Resharding" and
// Figure 4).  Under EP a rank holds E_local complete experts, W13
// [E_local, 2I, H] and W2 [E_local, H, I]; under TP every rank holds a 1/P
// shard of every expert, W13 [E, 2I/P, H] and W2 [E, H, I/P], the shards cut
// along the intermediate dimension (the output rows of W13, the input columns
// of W2).  EP -> TP packs one contiguous chunk per peer before the
// all-to-all, so the all-to-all lands every peer's shards in place; TP -> EP
// runs the inverse permute after the all-to-all.
//
// Chunk layout (one rank's buffer, peers outermost):
//   w13_chunks [P][E_local][2I/P][H]: for peer p and expert e, gate rows
//              [p*I/P, (p+1)*I/P) then up rows [I + p*I/P, I + (p+1)*I/P) --
//              itself a W13 of intermediate size I/P, gate rows first;
//   w2_chunks  [P][E_local][H][I/P]: columns [p*I/P, (p+1)*I/P) of every row.
//
// Both directions are one pass of 16-byte copies over contiguous segments (a
// W13 row of H elements, or I/P columns of a W2 row): HBM-bound, every byte
// read once and written once.
#include "moe_internal.cuh"

namespace moe {

namespace {

// Vector index arithmetic in 32 bits: the host checks that each weight
// tensor has fewer than 2^31 16-byte vectors.
struct ReshardShape {
  uint32_t E_l, H, I, P, Ip;
};

// Segment o of the chunk layout and the 16-byte vector where it starts in
// the EP layout.  W13: o = ((p*E_l + e)*2 + g)*Ip + r, a row of H elements;
// W2: o = (p*E_l + e)*H + h, Ip elements of row h.
__device__ __forceinline__ uint32_t ep_vector(const ReshardShape &s, bool w2, uint32_t o) {
  if (!w2) {
    const uint32_t r = o % s.Ip;
    uint32_t q = o / s.Ip;
    const uint32_t g = q & 1u;
    q >>= 1;
    const uint32_t e = q % s.E_l, p = q / s.E_l;
    return ((e * 2u + g) * s.I + p * s.Ip + r) * (s.H / 8u);
  }
  const uint32_t h = o % s.H;
  const uint32_t q = o / s.H;
  const uint32_t e = q % s.E_l, p = q / s.E_l;
  return (e * s.H + h) * (s.I / 8u) + p * (s.Ip / 8u);
}

// Vector i of one tensor's copy: its index in the source and in the
// destination (the chunk-layout side is sequential).
__device__ __forceinline__ void reshard_vector(const ReshardShape &s, bool w2, bool unpack,
                                               uint32_t i, uint32_t &from, uint32_t &to) {
  const uint32_t vps = (w2 ? s.Ip : s.H) / 8u;  // 16-byte vectors per segment
  const uint32_t o = i / vps, u = i - o * vps;
  const uint32_t ep = ep_vector(s, w2, o) + u;
  from = unpack ? i : ep;
  to = unpack ? ep : i;
}

// One launch copies both tensors: a grid-stride pass over W13's vectors,
// then W2's (a null tensor has none); kBatch vectors per thread are loaded
// before they are stored.
__global__ void __launch_bounds__(256)
    reshard_kernel(const uint4 *__restrict__ src13, uint4 *__restrict__ dst13,
                   const uint4 *__restrict__ src2, uint4 *__restrict__ dst2, ReshardShape s,
                   int unpack) {
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t n13 = src13 != nullptr ? s.E_l * 2u * s.I * (s.H / 8u) : 0u;
  const uint32_t n2 = src2 != nullptr ? s.E_l * s.H * (s.I / 8u) : 0u;
  const uint32_t total = n13 + n2;  // < 2^32: each is below 2^31
  const uint32_t stride = gridDim.x * blockDim.x;
  constexpr int kBatch = 4;
  for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += stride * kBatch) {
    uint4 v[kBatch];
    uint4 *d[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const uint32_t i = i0 + b * stride;  // no wrap: total + stride*kBatch < 2^32
      d[b] = nullptr;
      if (i < total) {
        const bool w2 = i >= n13;
        uint32_t from, to;
        reshard_vector(s, w2, unpack != 0, w2 ? i - n13 : i, from, to);
        v[b] = w2 ? src2[from] : src13[from];
        d[b] = w2 ? dst2 + to : dst13 + to;
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      if (d[b] != nullptr) *d[b] = v[b];
  }
}

}  // namespace

cudaError_t launch_reshard(int E_local, int H, int I, int P, const void *w13_src, void *w13_dst,
                           const void *w2_src, void *w2_dst, int unpack, cudaStream_t st) {
  ReshardShape s;
  s.E_l = (uint32_t)E_local;
  s.H = (uint32_t)H;
  s.I = (uint32_t)I;
  s.P = (uint32_t)P;
  s.Ip = (uint32_t)(I / P);
  const int grid = num_sms() * 8;
  cudaError_t e = launch_pdl(reshard_kernel, dim3(grid), dim3(256), 0, st,
                             static_cast<const uint4 *>(w13_src), static_cast<uint4 *>(w13_dst),
                             static_cast<const uint4 *>(w2_src), static_cast<uint4 *>(w2_dst), s,
                             unpack);
  return e;
}

}  // namespace moe
