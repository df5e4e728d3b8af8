// K0: the decoder's output projection fused with the first traversal.  In the LightSeq
// inference article (31duo.com, itemid-283120), hierarchical decoding section, the first
// traversal reads the [batch, beam, vocab] logits that the projection wrote; here the
// logits of a tile of 128 beams x 256 tokens are accumulated by the tensor cores in tensor
// memory and never stored.  The epilogue computes, per beam and chunk (1 to 4 sub-tiles of
// 256 tokens, the width chosen on the host), what K1 (beam_rows.cu) computes from stored
// logits -- the chunk max, the sum of exp(x - max), the group maxima -- and writes the
// chunk's candidates at or above its bound as slots, in the same record format; K2
// (beam_select.cu) finishes the step unchanged.
//
// One CTA per SM, in clusters of two CTAs that take adjacent 128-row blocks of the same
// chunk (so the pair reads each weight tile from L2 at about the same time), persistent
// over tiles of 2 x 128 rows x one chunk, 6 warps per CTA:
//   warp 0     TMA producer: a ring of [128 x kLgBK] hidden tiles and [256 x kLgBK] weight
//              tiles (f16 / bf16, swizzled rows of kLgBK elements), 192 KB in all, each CTA
//              loading its own tiles; the pair's first CTA prefetches the next sub-tile's
//              weight tile into L2;
//   warp 1     owns 512 tensor-memory columns; one lane issues tcgen05.mma (M 128, N 256,
//              K 16) into one of two 256-column accumulators, so one sub-tile's epilogue
//              overlaps the next sub-tile's products;
//   warps 2-5  epilogue: a thread is one beam (one tensor-memory lane).  Pass 1 reads its
//              256 accumulators of a sub-tile once: block and group maxima and the sum of
//              exp; pass 2 reads again only the blocks whose max reaches the bound and
//              stores the candidates from survivor bit masks.
// The bound is the larger of two lower bounds of the chunk's k-th largest x: the k-th
// largest group maximum and (k <= 8) the k-th largest 32-column block maximum.  A chunk
// keeps every candidate at or above its bound when they fit its slots, and otherwise its
// own top k (x descending, then token ascending), so the fine rank never needs the logits.
// Every wait is bounded: one that runs out sets the timeout bit of the status word, and the
// CTA lets its copies and products finish, frees its tensor memory and returns.
#include <cuda.h>

#include <climits>

#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr uint32_t kLgABytes = kLgM * kLgBK * 2;
constexpr uint32_t kLgBBytes = kLgN * kLgBK * 2;
constexpr int kLgStages = (192 * 1024) / (kLgABytes + kLgBBytes);
constexpr uint32_t kLgOffA = 0;
constexpr uint32_t kLgOffB = kLgOffA + kLgStages * kLgABytes;
constexpr uint32_t kLgOffBar = kLgOffB + kLgStages * kLgBBytes;
constexpr int kLgNumBars = 2 * kLgStages + 4 + 1;  // full, empty, tmem full x2, tmem empty x2, done
constexpr uint32_t kLgOffTmem = kLgOffBar + 8 * kLgNumBars;
constexpr uint32_t kLgOffAbort = kLgOffTmem + 4;
// pass 2 copies a lane's 32 values of a block to shared memory, rows of 36 floats (144
// bytes: 16-byte aligned, and 8 consecutive lanes' 16-byte stores hit distinct banks)
constexpr int kLgScratchStride = 36;
constexpr uint32_t kLgOffScratch = (kLgOffAbort + 4 + 15) & ~15u;
constexpr uint32_t kLgScratchBytes = 4 * 32 * kLgScratchStride * 4;
constexpr uint32_t kLgSmemUsed = kLgOffScratch + kLgScratchBytes;
constexpr size_t kLgSmemBytes = kLgSmemUsed + 1024;  // + alignment of the tiles to 1024 bytes
constexpr uint32_t kLgTmemCols = 2 * kLgN;
constexpr long long kLgDrainNs = 2000000000LL;
// sleep between polls of a waiting thread: the MMA lane reacts within ~30 ns to arrived data
// (a stage is ~280 ns of tensor work); the producer has 4 stages of slack
constexpr uint32_t kLgSleepMma = 32, kLgSleepProducer = 128, kLgSleepEpilogue = 64;
static_assert(kLgABytes % 1024 == 0 && kLgBBytes % 1024 == 0, "tiles must keep 1024-byte alignment");
static_assert(kLgBK * 2 == kLgSwizzleBytes, "a stage row is one swizzle row");

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

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
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
// Shared-memory matrix descriptor of a K-major tile written by TMA with the 128- or 64-byte
// swizzle: rows of kLgSwizzleBytes, 8-row swizzle atoms stacked along M / N.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);           // start address, 16-byte units
  d |= (uint64_t)1 << 16;                                       // leading-dimension offset (unused here)
  d |= (uint64_t)((8 * kLgSwizzleBytes) >> 4) << 32;            // stride between 8-row atoms
  d |= (uint64_t)1 << 46;                                       // descriptor version of tcgen05
  d |= (uint64_t)(kLgSwizzleBytes == 128 ? 2 : 4) << 61;        // 128- or 64-byte swizzle
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

// 64 consecutive fp32 columns of this thread's tensor-memory lane (two blocks), the load
// completed.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
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

// x of 32 accumulators of one row: + bias when there is one; columns at or past the
// vocab's end (n >= lim) become -inf.
template <bool BIAS, int N>
__device__ __forceinline__ void load_x(float (&v)[N], const float* bias, int col0, int lim) {
  if constexpr (BIAS) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] += i < lim ? __ldg(bias + col0 + i) : 0.0f;
  }
  if (lim < N) {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = i < lim ? v[i] : -INFINITY;
  }
}

// Bits i (i < 32) of the values v[off + i] >= R, in four independent chains; bits of columns
// at or past lim (the vocab's end) are clear.
template <int N>
__device__ __forceinline__ uint32_t survivor_mask(const float (&v)[N], int off, float R, int lim) {
  uint32_t m0 = 0, m1 = 0, m2 = 0, m3 = 0;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    m0 |= (v[off + i] >= R) ? (1u << i) : 0u;
    m1 |= (v[off + i + 1] >= R) ? (2u << i) : 0u;
    m2 |= (v[off + i + 2] >= R) ? (4u << i) : 0u;
    m3 |= (v[off + i + 3] >= R) ? (8u << i) : 0u;
  }
  uint32_t m = (m0 | m1) | (m2 | m3);
  if (lim < 32) m &= lim <= 0 ? 0u : (0xffffffffu >> (32 - lim));
  return m;
}

// Sub-tiles of chunk c: chunks of lp.sub_per_chunk sub-tiles, the last one shorter.
__device__ __forceinline__ int subtiles_of(const LogitsParams& lp, int c) {
  return min(lp.sub_per_chunk, lp.sub_per_row - c * lp.sub_per_chunk);
}

// L2 prefetch of a tensor-map box (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

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
  float* scratch_all = reinterpret_cast<float*>(gbase + kLgOffScratch);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.k, V = p.vocab, C = p.slot_cap, nc = p.nc;
  const int nk = (lp.dim + kLgBK - 1) / kLgBK;
  // tile t of cluster `cl`: chunk t / n_mp, 128-row block 2 (t % n_mp) + this CTA's rank
  const int n_mp = lp.n_mp, n_tiles = lp.n_tiles;
  const int crank = (int)cluster_ctarank(), cl = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);
  const long long spin = p.spin_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLgStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // this CTA's products are done before the stage refills
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
  // the fine rank may be scheduled from now on: its CTAs take the SMs this grid's CTAs leave
  // (they warm up, then wait for the whole grid before reading its records)
  grid_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t it = 0;
      bool ok = true, timed_out = false;
      for (int t = cl; t < n_tiles && ok; t += ncl) {
        const int mb = 2 * (t % n_mp) + crank, c = t / n_mp;
        const int nsub = subtiles_of(lp, c);
        for (int sub = 0; sub < nsub && ok; ++sub) {
          const int n0 = (c * lp.sub_per_chunk + sub) * kLgN;
          // the weight half of the next sub-tile this CTA multiplies, fetched into L2 while
          // this one runs (the first read of a weight tile otherwise waits on HBM)
          int n_next = -1;
          if (sub + 1 < nsub) {
            n_next = n0 + kLgN;
          } else if (t + ncl < n_tiles) {
            n_next = ((t + ncl) / n_mp) * lp.sub_per_chunk * kLgN;
          }
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = (int)(it % kLgStages);
            const uint32_t ph = (it / kLgStages) & 1u;
            if (!mbar_wait_sleep(empty_bar(s), ph ^ 1u, spin, kLgSleepProducer)) {
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
            if (n_next >= 0 && crank == 0) tma_prefetch_2d(&tmap_w, kb * kLgBK, n_next);
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
      for (int t = cl; t < n_tiles && ok; t += ncl) {
        const int c = t / n_mp;
        const int nsub = subtiles_of(lp, c);
        for (int sub = 0; sub < nsub && ok; ++sub, ++j) {
          const int buf = (int)(j & 1u);
          if (!mbar_wait_sleep(tempty_bar(buf), ((j >> 1) & 1u) ^ 1u, spin, kLgSleepMma)) {
            ok = false;
            timed_out = true;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)buf * kLgN;
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int s = (int)(it % kLgStages);
            if (!mbar_wait_sleep(full_bar(s), (it / kLgStages) & 1u, spin, kLgSleepMma) || *abort_flag) {
              timed_out = !*abort_flag;
              *abort_flag = 1;  // before the epilogue is released below
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a0 = kmajor_desc(sA + (uint32_t)s * kLgABytes);
            const uint64_t b0 = kmajor_desc(sB + (uint32_t)s * kLgBBytes);
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
    for (int t = cl; t < n_tiles && ok; t += ncl) {
      const int mb = 2 * (t % n_mp) + crank, c = t / n_mp;
      const int row = mb * kLgM + er;
      const bool live = row < p.rows && !(p.finished && p.finished[row]);
      const long long u = (long long)row * nc + c;
      CandSlot* slots = p.slots + u * C;
      const int nsub = subtiles_of(lp, c);
      float M = -INFINITY, S = 0.0f;
      float gm[G];
#pragma unroll
      for (int g = 0; g < G; ++g) gm[g] = -INFINITY;
      int nslot = 0;
      // the 8 largest 32-column block maxima of the chunk so far, descending
      float tb[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) tb[q] = -INFINITY;
      for (int sub = 0; sub < nsub; ++sub, ++j) {
        const int buf = (int)(j & 1u);
        if (!mbar_wait_sleep(tfull_bar(buf), (j >> 1) & 1u, spin, kLgSleepEpilogue)) {
          *abort_flag = 1;
          atomicOr(p.status, kDevTimeout);
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)buf * kLgN;
        const int n0 = (c * lp.sub_per_chunk + sub) * kLgN;
        const int lim = V - n0;  // columns of this sub-tile inside the vocab (> 0)
        auto xval = [&](float acc, int i) -> float {
          if constexpr (BIAS) return i < lim ? acc + __ldg(p.bias + n0 + i) : -INFINITY;
          return i < lim ? acc : -INFINITY;
        };
        // pass 1, one read of the accumulators: per 32-column block its group maxima (group =
        // column mod G) and max, and an online sum of exp(x - running max)
        constexpr int NB = kLgN / 32;
        float bmax[NB];
        float gs[G];
#pragma unroll
        for (int g = 0; g < G; ++g) gs[g] = -INFINITY;
        float ms = -INFINITY;
        float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
        const float2 L2 = make_float2(kLog2e, kLog2e);
#pragma unroll 1
        for (int jb = 0; jb < NB; ++jb) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)(jb * 32), v);
          load_x<BIAS, 32>(v, p.bias, n0 + jb * 32, lim - jb * 32);
          float gb[G];
#pragma unroll
          for (int g = 0; g < G; ++g) gb[g] = v[g];
#pragma unroll
          for (int i = G; i < 32; ++i) gb[i % G] = fmaxf(gb[i % G], v[i]);
          float bm = gb[0];
#pragma unroll
          for (int g = 1; g < G; ++g) bm = fmaxf(bm, gb[g]);
#pragma unroll
          for (int g = 0; g < G; ++g) gs[g] = fmaxf(gs[g], gb[g]);
          bmax[jb] = bm;
          const float mn = fmaxf(ms, bm);
          if (mn != -INFINITY) {
            if (mn != ms) {  // rescale the sum to the new running max (exact difference)
              const float r = fast_exp2((ms - mn) * kLog2e);
              acc0 = __fmul2_rn(acc0, make_float2(r, r));
              acc1 = __fmul2_rn(acc1, make_float2(r, r));
            }
            const float2 nm = make_float2(-mn, -mn);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float2 t0 = __fmul2_rn(__fadd2_rn(make_float2(v[i], v[i + 1]), nm), L2);
              const float2 t1 = __fmul2_rn(__fadd2_rn(make_float2(v[i + 2], v[i + 3]), nm), L2);
              acc0 = __fadd2_rn(acc0, make_float2(fast_exp2(t0.x), fast_exp2(t0.y)));
              acc1 = __fadd2_rn(acc1, make_float2(fast_exp2(t1.x), fast_exp2(t1.y)));
            }
          }
          ms = mn;
        }
        const float2 ap = __fadd2_rn(acc0, acc1);
        const float ss = ap.x + ap.y;  // sum over the sub-tile of exp(x - ms)
#pragma unroll
        for (int g = 0; g < G; ++g) gm[g] = fmaxf(gm[g], gs[g]);
        // bound: the k-th largest group maximum of the chunk so far, and for k <= 8 also the
        // k-th largest 32-column block maximum; each is at most the chunk's k-th largest x,
        // hence at most the row's, so every element of the row's top k passes the larger one
        // (blocks give a much tighter bound than k groups when one group's max is low)
#pragma unroll
        for (int jb = 0; jb < NB; ++jb) {
          float b = bmax[jb];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float hi = fmaxf(tb[q], b);
            b = fminf(tb[q], b);
            tb[q] = hi;
          }
        }
        float R = kth_of_groups<G>(gm, K);
        if (K <= 8) {
          float rb = -INFINITY;
#pragma unroll
          for (int q = 0; q < 8; ++q) rb = q == K - 1 ? tb[q] : rb;
          R = fmaxf(R, rb);
        }
        const float Mn = fmaxf(M, ms);
        if (Mn != -INFINITY) {
          S = (M == -INFINITY ? 0.0f : S * fast_exp2((M - Mn) * kLog2e)) +
              (ms == -INFINITY ? 0.0f : ss * fast_exp2((ms - Mn) * kLog2e));
        }
        M = Mn;
        // pass 2: the candidates x >= R, read again only for the blocks whose max reaches R
        // in some lane of the warp
        const int cap = C - K * (nsub - 1 - sub);  // leaves k slots for each later sub-tile
        const int n_before = nslot;
        const int room = live ? cap - n_before : 0;  // slots this sub-tile may fill
        int cnt = 0;
        float* scratch = scratch_all + (size_t)((warp - 2) * 32 + lane) * kLgScratchStride;
        uint32_t wmask = 0;  // blocks whose max reaches R
#pragma unroll
        for (int jb = 0; jb < NB; ++jb) wmask |= (bmax[jb] >= R) ? (1u << jb) : 0u;
        // the candidates of one block: copied to shared memory so that a column known only at
        // run time can be read back, then stored two at a time
        auto store_block = [&](uint32_t m, const float* vb, int col0) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(scratch + i) = make_float4(vb[i], vb[i + 1], vb[i + 2], vb[i + 3]);
          do {
            const int i0 = __ffs(m) - 1;
            m &= m - 1;
            const bool two = m != 0;
            const int i1 = two ? __ffs(m) - 1 : i0;
            m &= two ? m - 1 : m;
            const float x0 = scratch[i0], x1 = scratch[i1];
            if (cnt < room)
              *reinterpret_cast<float2*>(slots + n_before + cnt) = make_float2(x0, __int_as_float(col0 + i0));
            if (two && cnt + 1 < room)
              *reinterpret_cast<float2*>(slots + n_before + cnt + 1) = make_float2(x1, __int_as_float(col0 + i1));
            cnt += two ? 2 : 1;
          } while (m);
        };
        // two blocks at a time: one 64-column read, their masks computed together
#pragma unroll 1
        for (int jp = 0; jp < NB / 2; ++jp) {
          if (!__any_sync(0xffffffffu, (wmask >> (2 * jp)) & 3u)) continue;
          float v[64];
          tmem_ld64(taddr + (uint32_t)(jp * 64), v);
          const int c0 = jp * 64;
          load_x<BIAS, 64>(v, p.bias, n0 + c0, lim - c0);
          const uint32_t ma = survivor_mask<64>(v, 0, R, lim - c0);
          const uint32_t mb = survivor_mask<64>(v, 32, R, lim - c0 - 32);
          if (ma) store_block(ma, v, n0 + c0);
          if (mb) store_block(mb, v + 32, n0 + c0 + 32);
        }
        const bool over = n_before + cnt > cap;
        if (__any_sync(0xffffffffu, over)) {
          // too many candidates (ties): keep the sub-tile's own top k, in column order.  The
          // whole warp reads tensor memory; only the lanes that overflowed use the values.
          float px = INFINITY;
          int pc = -1;
          if (K <= 8) {
            // one pass: the 8 best keys in registers, sorted (x descending, then column
            // ascending), by insertion; the k-th of them is the threshold key
            float tx[8];
            int tc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              tx[q] = -INFINITY;
              tc[q] = INT_MAX;
            }
#pragma unroll 1
            for (int jb = 0; jb < kLgN / 32; ++jb) {
              float v[32];
              tmem_ld32(taddr + (uint32_t)(jb * 32), v);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int ci = jb * 32 + i, col = n0 + ci;
                const float x = xval(v[i], ci);
                if ((ci < lim) & ((x > tx[7]) | ((x == tx[7]) & (col < tc[7])))) {
                  tx[7] = x;
                  tc[7] = col;
#pragma unroll
                  for (int q = 7; q > 0; --q) {
                    const bool up = (tx[q] > tx[q - 1]) | ((tx[q] == tx[q - 1]) & (tc[q] < tc[q - 1]));
                    const float fx = up ? tx[q - 1] : tx[q];
                    const int fc = up ? tc[q - 1] : tc[q];
                    tx[q - 1] = up ? tx[q] : tx[q - 1];
                    tc[q - 1] = up ? tc[q] : tc[q - 1];
                    tx[q] = fx;
                    tc[q] = fc;
                  }
                }
              }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              px = q == K - 1 ? tx[q] : px;
              pc = q == K - 1 ? tc[q] : pc;
            }
          } else {
            // k > 8: k passes, each finding the next key in order
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

// Launch configuration: clusters of two CTAs, programmatic dependent launch.
struct PairLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  PairLaunch(int grid, cudaStream_t stream) : cfg{}, attr{} {
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kLgThreads);
    cfg.dynamicSmemBytes = kLgSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
  }
};

template <int G, bool BIAS>
cudaError_t launch_t(const CUtensorMap& mh, const CUtensorMap& mw, const LogitsParams& lp, int grid,
                     cudaStream_t stream) {
  PairLaunch l(grid, stream);
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

int logits_rows_max_clusters() {
  PairLaunch l(2, nullptr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, logits_rows_kernel<4, false>, &l.cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

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
