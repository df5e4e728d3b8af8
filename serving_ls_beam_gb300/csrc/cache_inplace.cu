// Beam-cache refresh in place, copy on change: cache[l, b*k+j, h, :len] becomes the old
// cache[l, b*k+parent[b,j], h, :len], touching only the rows whose parent is not themselves.
//
// Method: LightSeq inference article (31duo.com, itemid-283120) — after the fine rank
// "update the cache"; its latency breakdown puts the refresh at 10% (fp32) / 6% (fp16) of
// inference time.  The out-of-place refresh moves every row; here a row that continues
// itself is not moved at all, and a parent is read once for all the beams that continue it.
//
// GB300 design, three kernels (the host picks one):
//  * the bulk-copy kernel (aligned slabs, the long ones): one lane per CTA pipelines 1-D bulk
//    copies of the needed parents' slabs into shared memory and of the changed rows out;
//  * the word kernel (k <= 8, short slabs): a lane owns word positions and, per position,
//    loads every needed parent's word before writing any changed row;
//  * the staged CTA kernel (any shape): a persistent grid walks (layer, batch, head) units,
//    staging the needed parents' slabs in shared memory before writing the changed rows.
// In each, every row reads the state before the step, so swaps and cycles need no ordering
// and no global temporary.
#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr int kIpThreads = 512;
constexpr int kIpUnroll = 4;

template <int UNIT>
struct IpWord;
template <>
struct IpWord<16> {
  using T = uint4;
};
template <>
struct IpWord<8> {
  using T = uint2;
};
template <>
struct IpWord<4> {
  using T = uint32_t;
};
template <>
struct IpWord<2> {
  using T = uint16_t;
};
template <>
struct IpWord<1> {
  using T = uint8_t;
};

struct IpShared {
  int par[kMaxK];
  int slot[kMaxK];   // staging slot of each needed parent
  int nlist[kMaxK];  // needed parents, in row order
  int nneed;
  unsigned long long changed;  // bit j: row j takes another row's content
};

template <int UNIT>
__global__ void __launch_bounds__(kIpThreads) cache_inplace_kernel(const InplaceParams p) {
  using W = typename IpWord<UNIT>::T;
  extern __shared__ __align__(16) unsigned char ip_stage[];
  __shared__ IpShared sh;
  const int K = p.k, tid = threadIdx.x;
  const long long bh = (long long)p.batch * p.heads;
  grid_launch_dependents();
  grid_dependency_wait();  // the parents come from the beam step just before
  for (long long unit = blockIdx.x; unit < p.units; unit += gridDim.x) {
    const int l = (int)(unit / bh);
    const long long rem = unit - (long long)l * bh;
    const int b = (int)(rem / p.heads);
    const int h = (int)(rem - (long long)b * p.heads);
    __syncthreads();  // the previous unit is done with the staging space and sh
    if (tid < K) sh.par[tid] = __ldg(p.parent + b * K + tid);
    __syncthreads();
    if (tid == 0) {
      unsigned long long changed = 0, needed = 0;
      bool bad = false;
      for (int j = 0; j < K; ++j) {
        const int q = sh.par[j];
        if (q < 0 || q >= K) {
          bad = true;  // that row is left as it is
        } else if (q != j) {
          changed |= 1ull << j;
          needed |= 1ull << q;
        }
      }
      int n = 0;
      for (int q = 0; q < K; ++q)
        if ((needed >> q) & 1ull) {
          sh.slot[q] = n;
          sh.nlist[n++] = q;
        }
      sh.nneed = n;
      sh.changed = changed;
      if (bad && p.status) atomicOr(p.status, kDevBadParent);
    }
    __syncthreads();
    const unsigned long long changed = sh.changed;
    if (changed == 0ull) continue;  // CTA-uniform: nothing moves in this unit
    const int nneed = sh.nneed;
    // slab of row r: cache + l * layer_stride + (b*K + r) * row_stride + h * slab_stride
    unsigned char* unit_base = p.cache + (size_t)l * p.layer_stride + (size_t)b * K * p.row_stride +
                               (size_t)h * p.slab_stride;
    for (long long t0 = 0; t0 < p.slab_bytes; t0 += p.tile_bytes) {
      const int tb = (int)min((long long)p.tile_bytes, p.slab_bytes - t0);
      const int wpt = tb / UNIT;  // words per tile per row
      // stage the needed parents' tiles
      const int nload = nneed * wpt;
      for (int i0 = tid; i0 < nload; i0 += kIpThreads * kIpUnroll) {
        W w[kIpUnroll];
#pragma unroll
        for (int u = 0; u < kIpUnroll; ++u) {
          const int i = i0 + u * kIpThreads;
          if (i < nload) {
            const int s = i / wpt, e = i - s * wpt;
            w[u] = *reinterpret_cast<const W*>(unit_base + (size_t)sh.nlist[s] * p.row_stride + t0 + (size_t)e * UNIT);
          }
        }
#pragma unroll
        for (int u = 0; u < kIpUnroll; ++u) {
          const int i = i0 + u * kIpThreads;
          if (i < nload) reinterpret_cast<W*>(ip_stage)[i] = w[u];
        }
      }
      __syncthreads();
      // write the changed rows from the staged parents
      const int nstore = K * wpt;
      for (int i = tid; i < nstore; i += kIpThreads) {
        const int j = i / wpt, e = i - j * wpt;
        if ((changed >> j) & 1ull) {
          const int s = sh.slot[sh.par[j]];
          *reinterpret_cast<W*>(unit_base + (size_t)j * p.row_stride + t0 + (size_t)e * UNIT) =
              reinterpret_cast<const W*>(ip_stage)[s * wpt + e];
        }
      }
      __syncthreads();  // the staging space is reused by the next tile
    }
  }
}

// The same refresh driven by bulk (TMA) copies from one thread: a CTA is one warp whose
// lanes load the batches' parents into shared memory, after which lane 0 alone runs a
// two-stage pipeline over its (layer, batch, head group, tile) items, a step at a time: the
// bulk loads of the slabs step i needs are issued before the bulk stores of step i-1's changed
// rows, so a copy in each direction is always in flight.  A step takes as many of the item's
// heads as the slabs of the parents its batch actually needs fit a buffer (the host
// sizes items for a typical count of needed parents, not for all k).  Items differ in size (the rows a batch changes), so
// with a work counter (p.work) a CTA takes its next item when it is ready for one: the CTAs
// then finish together instead of with the sum of their items' sizes.  The last CTA to finish
// sets the counter back to zero for the next launch.  Requires 16-byte aligned slabs and
// tiles.
__global__ void __launch_bounds__(32) cache_inplace_tma_kernel(const InplaceParams p) {
  extern __shared__ __align__(128) unsigned char tsm[];
  __shared__ __align__(8) unsigned long long bar[2];
  const int K = p.k, lane = threadIdx.x;
  const int STAGE = p.stage_bytes;  // each of the two staging buffers
  int* par_s = reinterpret_cast<int*>(tsm + 2 * (size_t)STAGE);
  grid_launch_dependents();
  grid_dependency_wait();  // the parents come from the beam step just before
  for (int i = lane; i < p.batch * K; i += 32) par_s[i] = __ldg(p.parent + i);
  if (lane == 0) {
    mbar_init(smem_addr(&bar[0]), 1);
    mbar_init(smem_addr(&bar[1]), 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (lane != 0) return;  // lane 0 drives every copy from here on

  // an item: heads [h0, h0 + hg) of one (layer, batch), or one tile of one head's slabs
  const int HG = p.heads_per_item;
  const long long groups = (p.heads + HG - 1) / HG;
  const long long bg = (long long)p.batch * groups;
  const long long ntiles = (p.slab_bytes + p.tile_bytes - 1) / p.tile_bytes;
  uint32_t uses[2] = {0u, 0u};
  int cur = 0;
  bool bad = false, aborted = false;
  // the item whose loads are in flight and whose stores are still to be issued
  bool have_prev = false;
  unsigned char* pv_base = nullptr;
  unsigned long long pv_changed = 0, pv_needed = 0;
  int pv_b = 0, pv_tb = 0, pv_buf = 0, pv_hg = 0;
  uint32_t pv_parity = 0;

  auto finish_prev = [&]() {
    if (!mbar_wait_bounded(smem_addr(&bar[pv_buf]), pv_parity, p.spin_limit_ns)) {
      aborted = true;
      return;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const unsigned char* src = tsm + (size_t)pv_buf * STAGE;
    for (int j = 0; j < K; ++j) {
      if (!((pv_changed >> j) & 1ull)) continue;
      const int q = par_s[pv_b * K + j];
      const int slot = __popcll(pv_needed & ((1ull << q) - 1ull));
      for (int hh = 0; hh < pv_hg; ++hh)
        bulk_store(pv_base + (size_t)j * p.row_stride + (size_t)hh * p.slab_stride,
                   smem_addr(src + ((size_t)slot * pv_hg + hh) * pv_tb), (uint32_t)pv_tb);
    }
    bulk_commit();
  };

  const long long total = (long long)p.layers * bg * ntiles;
  uint32_t* const work = p.work;  // null: CTA c takes items c, c + grid, c + 2 grid, ...
  // the item after the current one, asked for one item ahead so that the atomic's latency
  // is hidden behind the current item's copies
  long long it = blockIdx.x;
  long long nxt = work ? (long long)gridDim.x + atomicAdd(work, 1u) : it + gridDim.x;
  while (it < total && !aborted) {
    const long long item = it;
    it = nxt;
    if (it < total) nxt = work ? (long long)gridDim.x + atomicAdd(work, 1u) : it + gridDim.x;
    const long long unit = item / ntiles;
    const long long tile = item - unit * ntiles;
    const int l = (int)(unit / bg);
    const long long rem = unit - (long long)l * bg;
    const int b = (int)(rem / groups);
    const int h0 = (int)(rem - (long long)b * groups) * HG;
    const int hg = min(HG, p.heads - h0);
    unsigned long long changed = 0, needed = 0;
    for (int j = 0; j < K; ++j) {
      const int q = par_s[b * K + j];
      if (q < 0 || q >= K) {
        bad = true;
      } else if (q != j) {
        changed |= 1ull << j;
        needed |= 1ull << q;
      }
    }
    if (changed == 0ull) continue;
    const long long t0 = tile * p.tile_bytes;
    const int tb = (int)min((long long)p.tile_bytes, p.slab_bytes - t0);
    // a step moves as many of the item's heads as the needed parents' slabs fit a buffer
    const int nn = __popcll(needed);
    const int hsub = max(1, min(hg, STAGE / (nn * tb)));
    for (int hs = 0; hs < hg && !aborted; hs += hsub) {
      const int hn = min(hsub, hg - hs);
      unsigned char* base = p.cache + (size_t)l * p.layer_stride + (size_t)b * K * p.row_stride +
                            (size_t)(h0 + hs) * p.slab_stride + t0;
      // buffer `cur` was last read by the stores of the step before the previous one
      bulk_wait_read<0>();
      const uint32_t b_addr = smem_addr(&bar[cur]);
      mbar_arrive_expect_tx(b_addr, (uint32_t)(nn * hn * tb));
      unsigned char* dst = tsm + (size_t)cur * STAGE;
      int slot = 0;
      for (int q = 0; q < K; ++q) {
        if (!((needed >> q) & 1ull)) continue;
        for (int hh = 0; hh < hn; ++hh)
          bulk_load_plain(smem_addr(dst + ((size_t)slot * hn + hh) * tb),
                          base + (size_t)q * p.row_stride + (size_t)hh * p.slab_stride, (uint32_t)tb, b_addr);
        ++slot;
      }
      if (have_prev) finish_prev();
      have_prev = true;
      pv_base = base;
      pv_changed = changed;
      pv_needed = needed;
      pv_b = b;
      pv_tb = tb;
      pv_hg = hn;
      pv_buf = cur;
      pv_parity = uses[cur] & 1u;
      ++uses[cur];
      cur ^= 1;
    }
  }
  if (have_prev && !aborted) finish_prev();
  if (aborted) {
    // a wait ran out: record it, and let the copies in flight land before leaving
    if (p.status) atomicOr(p.status, kDevTimeout);
    for (int s = 0; s < 2; ++s)
      if (uses[s] > 0) mbar_wait_bounded(smem_addr(&bar[s]), (uses[s] - 1) & 1u, 2000000000LL);
  }
  bulk_wait_all();
  if (bad && p.status) atomicOr(p.status, kDevBadParent);
  if (work) {
    // every CTA has taken its last item once all have counted themselves out here
    __threadfence();
    if (atomicAdd(work + 1, 1u) == gridDim.x - 1u) {
      work[0] = 0u;
      work[1] = 0u;
    }
  }
}

// The same refresh by plain word copies, for k <= KT: a warp takes an item (heads
// [h0, h0 + word_heads) of one (layer, batch)), and each lane owns a set of word positions in
// it.  For a position, the lane first loads that word of every needed parent into registers,
// then writes it to every changed row whose parent it is.  A word position belongs to one lane
// in every row of the item, so rows that are both read and overwritten (swaps, cycles) need
// no staging, no barrier and no ordering between lanes.  U positions are in flight per lane.
template <int KT, int UNIT>
__global__ void __launch_bounds__(kIpWordThreads) cache_inplace_words_kernel(const InplaceParams p) {
  using Wd = typename IpWord<UNIT>::T;
  constexpr int U = KT <= 4 ? 4 : 2;  // word positions per lane and round
  const int K = p.k, lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * kIpWordThreads + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * kIpWordThreads) >> 5;
  extern __shared__ int wpar[];  // every batch's parents, [batch * k]
  const int HG = p.word_heads;
  const long long groups = (p.heads + HG - 1) / HG;
  const long long bg = (long long)p.batch * groups;
  grid_launch_dependents();
  grid_dependency_wait();  // the parents come from the beam step just before
  for (int i = threadIdx.x; i < p.batch * K; i += kIpWordThreads) wpar[i] = __ldg(p.parent + i);
  __syncthreads();
  bool bad = false;
  for (long long item = warp0; item < p.word_items; item += nwarps) {
    const int l = (int)(item / bg);
    const long long rem = item - (long long)l * bg;
    const int b = (int)(rem / groups);
    const int h0 = (int)(rem - (long long)b * groups) * HG;
    const int hg = min(HG, p.heads - h0);
    // the batch's parents: which rows change (changed) and, per parent q, the rows it feeds
    const int myq = lane < K ? wpar[b * K + lane] : lane;
    unsigned tgt[KT];
#pragma unroll
    for (int q = 0; q < KT; ++q) tgt[q] = 0u;
    unsigned changed = 0u;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      const int q = __shfl_sync(0xffffffffu, myq, j);
      if (j < K) {
        if (q < 0 || q >= K) {
          bad = true;  // that row is left as it is
        } else if (q != j) {
          changed |= 1u << j;
#pragma unroll
          for (int qq = 0; qq < KT; ++qq) tgt[qq] |= (qq == q ? 1u : 0u) << j;
        }
      }
    }
    if (changed == 0u) continue;  // warp-uniform: nothing moves in this item
    unsigned char* base = p.cache + (size_t)l * p.layer_stride + (size_t)b * K * p.row_stride +
                          (size_t)h0 * p.slab_stride;
    const uint32_t nw = (uint32_t)(hg * p.slab_words);
    for (uint32_t w0 = lane; w0 < nw; w0 += 32 * U) {
      Wd v[U][KT];
      size_t off[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t w = w0 + 32u * u;
        const uint32_t h = fast_div(w, p.word_magic, p.word_shift);
        const uint32_t e = w - h * (uint32_t)p.slab_words;
        off[u] = (size_t)h * p.slab_stride + (size_t)e * UNIT;
        if (w < nw) {
#pragma unroll
          for (int q = 0; q < KT; ++q)
            if (tgt[q]) v[u][q] = *reinterpret_cast<const Wd*>(base + (size_t)q * p.row_stride + off[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (w0 + 32u * u < nw) {
#pragma unroll
          for (int q = 0; q < KT; ++q) {
            unsigned m = tgt[q];
            while (m) {
              const int j = __ffs(m) - 1;
              m &= m - 1u;
              *reinterpret_cast<Wd*>(base + (size_t)j * p.row_stride + off[u]) = v[u][q];
            }
          }
        }
      }
    }
  }
  if (bad && lane == 0 && p.status) atomicOr(p.status, kDevBadParent);
}

size_t words_smem(int batch, int k) { return align_up((size_t)batch * k * sizeof(int32_t), 16); }

template <int KT, int UNIT>
cudaError_t launch_w(const InplaceParams& p, int grid, cudaStream_t stream) {
  PdlLaunch l(dim3((unsigned)grid), dim3(kIpWordThreads), words_smem(p.batch, p.k), stream);
  return cudaLaunchKernelEx(&l.cfg, cache_inplace_words_kernel<KT, UNIT>, p);
}

template <int UNIT>
cudaError_t launch_u(const InplaceParams& p, int grid, size_t smem, cudaStream_t stream) {
  PdlLaunch l(dim3((unsigned)grid), dim3(kIpThreads), smem, stream);
  return cudaLaunchKernelEx(&l.cfg, cache_inplace_kernel<UNIT>, p);
}

template <int UNIT>
cudaError_t config_u(size_t smem, int* occ) {
  cudaError_t e =
      cudaFuncSetAttribute(cache_inplace_kernel<UNIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, cache_inplace_kernel<UNIT>, kIpThreads, smem);
}

}  // namespace

size_t cache_inplace_tma_smem(int stage_bytes, int batch, int k) {
  return 2 * (size_t)stage_bytes + align_up((size_t)batch * k * sizeof(int32_t), 16);
}

cudaError_t launch_cache_inplace_tma(const InplaceParams& p, int grid, cudaStream_t stream) {
  PdlLaunch l(dim3((unsigned)grid), dim3(32), cache_inplace_tma_smem(p.stage_bytes, p.batch, p.k), stream);
  return cudaLaunchKernelEx(&l.cfg, cache_inplace_tma_kernel, p);
}

cudaError_t cache_inplace_tma_occupancy(int stage_bytes, int batch, int k, int* occ) {
  const size_t smem = cache_inplace_tma_smem(stage_bytes, batch, k);
  cudaError_t e = cudaFuncSetAttribute(cache_inplace_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, cache_inplace_tma_kernel, 32, smem);
}

cudaError_t launch_cache_inplace(const InplaceParams& p, int unit, int grid, cudaStream_t stream) {
  const size_t smem = (size_t)kIpStageBytes;
  switch (unit) {
    case 16: return launch_u<16>(p, grid, smem, stream);
    case 8: return launch_u<8>(p, grid, smem, stream);
    case 4: return launch_u<4>(p, grid, smem, stream);
    case 2: return launch_u<2>(p, grid, smem, stream);
    case 1: return launch_u<1>(p, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_cache_inplace_words(const InplaceParams& p, int unit, int grid, cudaStream_t stream) {
  const bool k4 = p.k <= 4;
  switch (unit) {
    case 16: return k4 ? launch_w<4, 16>(p, grid, stream) : launch_w<8, 16>(p, grid, stream);
    case 8: return k4 ? launch_w<4, 8>(p, grid, stream) : launch_w<8, 8>(p, grid, stream);
    case 4: return k4 ? launch_w<4, 4>(p, grid, stream) : launch_w<8, 4>(p, grid, stream);
    case 2: return k4 ? launch_w<4, 2>(p, grid, stream) : launch_w<8, 2>(p, grid, stream);
    case 1: return k4 ? launch_w<4, 1>(p, grid, stream) : launch_w<8, 1>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int KT, int UNIT>
cudaError_t occ_w(int batch, int k, int* occ) {
  const size_t smem = words_smem(batch, k);
  cudaError_t e = cudaFuncSetAttribute(cache_inplace_words_kernel<KT, UNIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, cache_inplace_words_kernel<KT, UNIT>, kIpWordThreads,
                                                       smem);
}

cudaError_t cache_inplace_words_occupancy(int unit, int batch, int k, int* occ) {
  const bool k4 = k <= 4;
  switch (unit) {
    case 16: return k4 ? occ_w<4, 16>(batch, k, occ) : occ_w<8, 16>(batch, k, occ);
    case 8: return k4 ? occ_w<4, 8>(batch, k, occ) : occ_w<8, 8>(batch, k, occ);
    case 4: return k4 ? occ_w<4, 4>(batch, k, occ) : occ_w<8, 4>(batch, k, occ);
    case 2: return k4 ? occ_w<4, 2>(batch, k, occ) : occ_w<8, 2>(batch, k, occ);
    case 1: return k4 ? occ_w<4, 1>(batch, k, occ) : occ_w<8, 1>(batch, k, occ);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t cache_inplace_occupancy(int unit, int* occ) {
  const size_t smem = (size_t)kIpStageBytes;
  switch (unit) {
    case 16: return config_u<16>(smem, occ);
    case 8: return config_u<8>(smem, occ);
    case 4: return config_u<4>(smem, occ);
    case 2: return config_u<2>(smem, occ);
    case 1: return config_u<1>(smem, occ);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsb
