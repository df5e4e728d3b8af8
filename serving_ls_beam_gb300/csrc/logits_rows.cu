// K0: the decoder's output projection fused with the first traversal.  In the LightSeq
// inference article (31duo.com, itemid-283120), hierarchical decoding section, the first
// traversal reads the [batch, beam, vocab] logits that the projection wrote; here the
// logits of a tile of 128 beams x 256 tokens are accumulated by the tensor cores in tensor
// memory and never stored.  The tile's epilogue computes, per beam and 512-token chunk,
// what K1 (beam_rows.cu) computes from stored logits -- the chunk max, the sum of
// exp(x - max), the group maxima -- and writes the chunk's candidates at or above its
// R-top-k bound as slots, in the same record format; K2 (beam_select.cu) finishes the
// step unchanged.
//
// One CTA per SM, persistent over tiles of 128 rows x 512 columns (a chunk), 6 warps:
//   warp 0     TMA producer: a 4-stage ring of [128 x 64] hidden and [256 x 64] weight
//              tiles (f16 / bf16, 128-byte swizzle), one stage per 64 of the hidden size;
//   warp 1     owns 512 tensor-memory columns; one lane issues tcgen05.mma (M 128, N 256,
//              K 16) into one of two 256-column accumulators, so one sub-tile's epilogue
//              overlaps the next sub-tile's products;
//   warps 2-5  epilogue: a thread is one beam (one tensor-memory lane); it reads its 256
//              accumulators of a sub-tile twice: max and group maxima, then the sum of exp
//              and the candidates at or above the bound.
// A chunk keeps every candidate at or above its bound when they fit its slots, and
// otherwise its own top k (x descending, then token ascending), so the fine rank never
// needs the logits.  Every wait is bounded: one that runs out sets the timeout bit of the
// status word, and the CTA lets its copies and products finish, frees its tensor memory
// and returns.
#include <cuda.h>

#include <climits>

#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr int kLgStages = 4;
constexpr uint32_t kLgABytes = kLgM * kLgBK * 2;  // 16 KB
constexpr uint32_t kLgBBytes = kLgN * kLgBK * 2;  // 32 KB
constexpr uint32_t kLgOffA = 0;
constexpr uint32_t kLgOffB = kLgOffA + kLgStages * kLgABytes;
constexpr uint32_t kLgOffBar = kLgOffB + kLgStages * kLgBBytes;
constexpr int kLgNumBars = 2 * kLgStages + 4 + 1;  // full, empty, tmem full x2, tmem empty x2, done
constexpr uint32_t kLgOffTmem = kLgOffBar + 8 * kLgNumBars;
constexpr uint32_t kLgOffAbort = kLgOffTmem + 4;
constexpr uint32_t kLgSmemUsed = kLgOffAbort + 4;
constexpr size_t kLgSmemBytes = kLgSmemUsed + 1024;  // + alignment of the tiles to 1024 bytes
constexpr uint32_t kLgTmemCols = 2 * kLgN;
constexpr long long kLgDrainNs = 2000000000LL;
static_assert(kLgABytes % 1024 == 0 && kLgBBytes % 1024 == 0, "tiles must keep 1024-byte alignment");
static_assert(kLgBK * 2 == 128, "one stage row is one 128-byte swizzle row");

// ---------------------------------------------------------------- tcgen05 / TMA helpers
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] . B[smem]^T, both K-major; accumulate unless acc == 0.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along M / N.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, 16-byte units
  d |= (uint64_t)1 << 16;                              // leading-dimension offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                    // stride between 8-row atoms
  d |= (uint64_t)1 << 46;                              // descriptor version of tcgen05
  d |= (uint64_t)2 << 61;                              // 128-byte swizzle
  return d;
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane, the load completed.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  __syncwarp();  // the load is warp-wide (.sync.aligned)
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// k-th largest (1-based) of the G group maxima; ties by group index.  With k = G it is
// the least of them.
template <int G>
__device__ __forceinline__ float kth_of_groups(const float (&gm)[G], int k) {
  if (k == G) {
    float r = gm[0];
#pragma unroll
    for (int g = 1; g < G; ++g) r = fminf(r, gm[g]);
    return r;
  }
  float R = -INFINITY;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    int rank = 0;
#pragma unroll
    for (int h = 0; h < G; ++h) rank += (gm[h] > gm[g]) | ((gm[h] == gm[g]) & (h < g));
    R = rank == k - 1 ? gm[g] : R;
  }
  return R;
}

__device__ __forceinline__ int subtiles_of(int c, int vocab) { return c * kLgChunk + kLgN < vocab ? 2 : 1; }

template <int G, bool BIAS>
__global__ void __launch_bounds__(kLgThreads, 1)
    logits_rows_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
                       const LogitsParams lp) {
  const StepParams& p = lp.s;
  extern __shared__ unsigned char lg_smem_raw[];
  const uint32_t raw = smem_addr(lg_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = lg_smem_raw + (base - raw);
  const uint32_t sA = base + kLgOffA, sB = base + kLgOffB, bar0 = base + kLgOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(kLgStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kLgStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kLgStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (uint32_t)(2 * kLgStages + 4);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + kLgOffTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kLgOffAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.k, V = p.vocab, C = p.slot_cap, nc = p.nc;
  const int nk = (lp.dim + kLgBK - 1) / kLgBK;
  const int n_m = lp.n_m, n_tiles = lp.n_tiles;
  const long long spin = p.spin_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLgStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);  // one arrival per epilogue warp
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(base + kLgOffTmem, kLgTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the hidden states may come from the previous kernel of the stream
  grid_dependency_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t it = 0;
      bool ok = true, timed_out = false;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int mb = t % n_m, c = t / n_m;
        const int nsub = subtiles_of(c, V);
        for (int sub = 0; sub < nsub && ok; ++sub) {
          const int n0 = c * kLgChunk + sub * kLgN;
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = (int)(it % kLgStages);
            const uint32_t ph = (it / kLgStages) & 1u;
            if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, spin)) {
              ok = false;
              timed_out = true;
              break;
            }
            if (*abort_flag) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full_bar(s), kLgABytes + kLgBBytes);
            tma_load_2d(sA + (uint32_t)s * kLgABytes, &tmap_h, kb * kLgBK, mb * kLgM, full_bar(s));
            tma_load_2d(sB + (uint32_t)s * kLgBBytes, &tmap_w, kb * kLgBK, n0, full_bar(s));
          }
        }
      }
      if (timed_out) {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
      }
      // every copy issued lands before the CTA may exit
      for (uint32_t n = it > (uint32_t)kLgStages ? it - kLgStages : 0u; n < it; ++n)
        mbar_wait_bounded(full_bar((int)(n % kLgStages)), (n / kLgStages) & 1u, kLgDrainNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t idesc = lp.idesc;
      uint32_t it = 0, j = 0;
      bool ok = true, timed_out = false;
      for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
        const int c = t / n_m;
        const int nsub = subtiles_of(c, V);
        for (int sub = 0; sub < nsub && ok; ++sub, ++j) {
          const int buf = (int)(j & 1u);
          if (!mbar_wait_bounded(tempty_bar(buf), ((j >> 1) & 1u) ^ 1u, spin)) {
            ok = false;
            timed_out = true;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)buf * kLgN;
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = (int)(it % kLgStages);
            if (!mbar_wait_bounded(full_bar(s), (it / kLgStages) & 1u, spin) || *abort_flag) {
              timed_out = !*abort_flag;
              *abort_flag = 1;  // before the epilogue is released below
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a0 = sw128_desc(sA + (uint32_t)s * kLgABytes);
            const uint64_t b0 = sw128_desc(sB + (uint32_t)s * kLgBBytes);
#pragma unroll
            for (int kk = 0; kk < kLgBK / 16; ++kk)  // 16 elements = 32 bytes along the swizzled row
              umma_f16(d, a0 + 2u * kk, b0 + 2u * kk, idesc, (uint32_t)((kb | kk) != 0));
            umma_commit(empty_bar(s));  // the stage is free once these products are done
          }
          if (!ok) {
            umma_commit(tfull_bar(buf));  // release the epilogue; it sees the abort flag
            break;
          }
          umma_commit(tfull_bar(buf));
        }
      }
      if (timed_out) {
        *abort_flag = 1;
        atomicOr(p.status, kDevTimeout);
      }
      umma_commit(done_bar);
      mbar_wait_bounded(done_bar, 0u, kLgDrainNs);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // the tensor-memory lane quarter this warp may access
    const int er = q * 32 + lane;
    uint32_t j = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const int mb = t % n_m, c = t / n_m;
      const int row = mb * kLgM + er;
      const bool live = row < p.rows && !(p.finished && p.finished[row]);
      const long long u = (long long)row * nc + c;
      CandSlot* slots = p.slots + u * C;
      const int nsub = subtiles_of(c, V);
      float M = -INFINITY, S = 0.0f;
      float gm[G];
#pragma unroll
      for (int g = 0; g < G; ++g) gm[g] = -INFINITY;
      int nslot = 0;
      for (int sub = 0; sub < nsub; ++sub, ++j) {
        const int buf = (int)(j & 1u);
        if (!mbar_wait_bounded(tfull_bar(buf), (j >> 1) & 1u, spin)) {
          *abort_flag = 1;
          atomicOr(p.status, kDevTimeout);
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)buf * kLgN;
        const int n0 = c * kLgChunk + sub * kLgN;
        const int lim = V - n0;  // columns of this sub-tile inside the vocab (> 0)
        auto xval = [&](float acc, int i) -> float {
          if constexpr (BIAS) return i < lim ? acc + __ldg(p.bias + n0 + i) : -INFINITY;
          return i < lim ? acc : -INFINITY;
        };
        // pass 1: group maxima of the sub-tile (group = column mod G)
        float gs[G];
#pragma unroll
        for (int g = 0; g < G; ++g) gs[g] = -INFINITY;
#pragma unroll 1
        for (int jb = 0; jb < kLgN / 32; ++jb) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)(jb * 32), v);
#pragma unroll
          for (int i = 0; i < 32; ++i) gs[i % G] = fmaxf(gs[i % G], xval(v[i], jb * 32 + i));
        }
        float ms = gs[0];
#pragma unroll
        for (int g = 1; g < G; ++g) ms = fmaxf(ms, gs[g]);
#pragma unroll
        for (int g = 0; g < G; ++g) gm[g] = fmaxf(gm[g], gs[g]);
        // bound: k-th largest group maximum of the chunk so far (never above the chunk's
        // k-th largest x, so every candidate of the final top k passes it)
        const float R = kth_of_groups<G>(gm, K);
        const float Mn = fmaxf(M, ms);
        if (M != -INFINITY) S *= fast_exp2((M - Mn) * kLog2e);
        M = Mn;
        // pass 2: sum of exp(x - M) and the candidates x >= R
        const int cap = (sub == 0 && nsub == 2) ? C - K : C;  // leaves k slots for the second half
        const int n_before = nslot;
        int cnt = 0;
        float ssum = 0.0f;
#pragma unroll 1
        for (int jb = 0; jb < kLgN / 32; ++jb) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)(jb * 32), v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int ci = jb * 32 + i;
            const float x = xval(v[i], ci);
            if (M != -INFINITY) ssum += fast_exp2((x - M) * kLog2e);
            if (ci < lim && x >= R) {
              if (live && n_before + cnt < cap) {
                CandSlot cs;
                cs.x = x;
                cs.v = n0 + ci;
                slots[n_before + cnt] = cs;
              }
              ++cnt;
            }
          }
        }
        S += ssum;
        const bool over = n_before + cnt > cap;
        if (__any_sync(0xffffffffu, over)) {
          // too many candidates (ties): keep the sub-tile's own top k, in column order.  The
          // whole warp reads tensor memory; only the lanes that overflowed use the values.
          float px = INFINITY;
          int pc = -1;
          for (int r = 0; r < K; ++r) {
            float bx = -INFINITY;
            int bc = INT_MAX;
#pragma unroll 1
            for (int jb = 0; jb < kLgN / 32; ++jb) {
              float v[32];
              tmem_ld32(taddr + (uint32_t)(jb * 32), v);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int ci = jb * 32 + i, col = n0 + ci;
                const float x = xval(v[i], ci);
                const bool after_prev = (x < px) | ((x == px) & (col > pc));
                const bool before_best = (x > bx) | ((x == bx) & (col < bc));
                if ((ci < lim) & after_prev & before_best) {
                  bx = x;
                  bc = col;
                }
              }
            }
            px = bx;
            pc = bc;
          }
          int n = n_before;
#pragma unroll 1
          for (int jb = 0; jb < kLgN / 32; ++jb) {
            float v[32];
            tmem_ld32(taddr + (uint32_t)(jb * 32), v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int ci = jb * 32 + i, col = n0 + ci;
              const float x = xval(v[i], ci);
              if (over && (ci < lim) && ((x > px) | ((x == px) & (col <= pc)))) {
                if (live) {
                  CandSlot cs;
                  cs.x = x;
                  cs.v = col;
                  slots[n] = cs;
                }
                ++n;
              }
            }
          }
          if (over) cnt = n - n_before;
        }
        nslot = n_before + cnt;
        // the accumulators of this sub-tile are no longer needed
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      }
      if (!ok) break;
      if (live) {
        float* rec = reinterpret_cast<float*>(p.rec + (size_t)u * p.rec_stride);
        *reinterpret_cast<float4*>(rec) = make_float4(__int_as_float(nslot), M, S, 0.0f);
        if constexpr (G >= 4) {
#pragma unroll
          for (int g = 0; g < G; g += 4)
            *reinterpret_cast<float4*>(rec + 4 + g) = make_float4(gm[g], gm[g + 1], gm[g + 2], gm[g + 3]);
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) rec[4 + g] = gm[g];
        }
      }
    }
  }
  // teardown: every product and tensor-memory read is done before the columns are freed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kLgTmemCols);
  }
}

template <int G, bool BIAS>
cudaError_t launch_t(const CUtensorMap& mh, const CUtensorMap& mw, const LogitsParams& lp, int grid,
                     cudaStream_t stream) {
  PdlLaunch l(dim3((unsigned)grid), dim3(kLgThreads), kLgSmemBytes, stream);
  return cudaLaunchKernelEx(&l.cfg, logits_rows_kernel<G, BIAS>, mh, mw, lp);
}

template <int G>
cudaError_t config_g() {
  cudaError_t e = cudaFuncSetAttribute(logits_rows_kernel<G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kLgSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_rows_kernel<G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kLgSmemBytes);
  return e;
}

}  // namespace

size_t logits_rows_smem_bytes() { return kLgSmemBytes; }

cudaError_t logits_rows_config() {
  cudaError_t e = config_g<1>();
  if (e == cudaSuccess) e = config_g<2>();
  if (e == cudaSuccess) e = config_g<4>();
  if (e == cudaSuccess) e = config_g<8>();
  if (e == cudaSuccess) e = config_g<16>();
  if (e == cudaSuccess) e = config_g<32>();
  return e;
}

cudaError_t launch_logits_rows(const CUtensorMap& mh, const CUtensorMap& mw, const LogitsParams& lp, int grid,
                               cudaStream_t stream) {
  const bool bias = lp.s.bias != nullptr;
  switch (lp.s.groups) {
    case 1: return bias ? launch_t<1, true>(mh, mw, lp, grid, stream) : launch_t<1, false>(mh, mw, lp, grid, stream);
    case 2: return bias ? launch_t<2, true>(mh, mw, lp, grid, stream) : launch_t<2, false>(mh, mw, lp, grid, stream);
    case 4: return bias ? launch_t<4, true>(mh, mw, lp, grid, stream) : launch_t<4, false>(mh, mw, lp, grid, stream);
    case 8: return bias ? launch_t<8, true>(mh, mw, lp, grid, stream) : launch_t<8, false>(mh, mw, lp, grid, stream);
    case 16:
      return bias ? launch_t<16, true>(mh, mw, lp, grid, stream) : launch_t<16, false>(mh, mw, lp, grid, stream);
    case 32:
      return bias ? launch_t<32, true>(mh, mw, lp, grid, stream) : launch_t<32, false>(mh, mw, lp, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsb
