// Beam-cache refresh: gather the [layers, batch*k, heads, max_len, head_dim] cache
// by parent beam, positions [0, len) only.
//
// Method: LightSeq inference article (31duo.com, itemid-283120) — after the fine rank
// "update the cache"; its latency breakdown figure puts the refresh at 10% (fp32) /
// 6% (fp16) of inference time.  This is pure HBM streaming: every byte is read once
// and written once.  A persistent grid walks (layer, row) pairs; each pair is heads
// slabs of len*head_dim elements at a fixed stride, copied as UNIT-byte words with
// several independent loads in flight per thread before the stores.
#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr int kCopyThreads = 512;
constexpr int kUnroll = 4;

template <int UNIT>
struct Word;
template <>
struct Word<16> {
  using T = uint4;
};
template <>
struct Word<8> {
  using T = uint2;
};
template <>
struct Word<4> {
  using T = uint32_t;
};
template <>
struct Word<2> {
  using T = uint16_t;
};
template <>
struct Word<1> {
  using T = uint8_t;
};

template <int UNIT>
__global__ void __launch_bounds__(kCopyThreads) cache_reorder_kernel(const ReorderParams p) {
  using W = typename Word<UNIT>::T;
  const uint32_t per_pair = (uint32_t)p.slab_units * (uint32_t)p.heads;
  grid_launch_dependents();
  grid_dependency_wait();  // the parents come from the beam step just before
  for (long long pair = blockIdx.x; pair < p.pairs; pair += gridDim.x) {
    const int l = (int)(pair / p.rows);
    const int r = (int)(pair - (long long)l * p.rows);
    const int par = __ldg(p.parent + r);
    if (par < 0 || par >= p.k) {
      if (threadIdx.x == 0 && p.status) atomicOr(p.status, kDevBadParent);
      continue;
    }
    const int srow = (r / p.k) * p.k + par;
    const unsigned char* src = p.src + (size_t)l * p.layer_stride + (size_t)srow * p.row_stride;
    unsigned char* dst = p.dst + (size_t)l * p.layer_stride + (size_t)r * p.row_stride;
    for (uint32_t base = threadIdx.x; base < per_pair; base += kCopyThreads * kUnroll) {
      W w[kUnroll];
      size_t off[kUnroll];
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const uint32_t i = base + t * kCopyThreads;
        const uint32_t h = fast_div(i, p.div_units_magic, p.div_units_shift);
        const uint32_t e = i - h * (uint32_t)p.slab_units;
        off[t] = (size_t)h * p.slab_stride + (size_t)e * UNIT;
        if (i < per_pair) w[t] = *reinterpret_cast<const W*>(src + off[t]);
      }
#pragma unroll
      for (int t = 0; t < kUnroll; ++t) {
        const uint32_t i = base + t * kCopyThreads;
        if (i < per_pair) *reinterpret_cast<W*>(dst + off[t]) = w[t];
      }
    }
  }
}

template <int UNIT>
cudaError_t launch_u(const ReorderParams& p, int grid, cudaStream_t stream) {
  PdlLaunch l(dim3((unsigned)grid), dim3(kCopyThreads), 0, stream);
  return cudaLaunchKernelEx(&l.cfg, cache_reorder_kernel<UNIT>, p);
}

template <int UNIT>
cudaError_t occ_u(int* occ) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, cache_reorder_kernel<UNIT>, kCopyThreads, 0);
}

}  // namespace

cudaError_t launch_cache_reorder(const ReorderParams& p, int unit, int grid, cudaStream_t stream) {
  switch (unit) {
    case 16: return launch_u<16>(p, grid, stream);
    case 8: return launch_u<8>(p, grid, stream);
    case 4: return launch_u<4>(p, grid, stream);
    case 2: return launch_u<2>(p, grid, stream);
    case 1: return launch_u<1>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t cache_reorder_occupancy(int unit, int* occ) {
  switch (unit) {
    case 16: return occ_u<16>(occ);
    case 8: return occ_u<8>(occ);
    case 4: return occ_u<4>(occ);
    case 2: return occ_u<2>(occ);
    case 1: return occ_u<1>(occ);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsb
