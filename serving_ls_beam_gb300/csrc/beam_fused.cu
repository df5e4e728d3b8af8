// Beam-step kernel K3: the whole step of one batch in one CTA -- both traversals of the
// batch's beams and the fine rank -- for batches that fill the GPU on their own.  The same
// kernel is the one-kernel sampler of sampling decoding (SAMP): a CTA takes kFuSampRows
// independent rows, and per row the candidates at or above its bound give its exact top k,
// from which one token is drawn at the caller's uniform (ls_draw.cuh).
//
// Method: LightSeq inference article (31duo.com, itemid-283120), hierarchical decoding
// section.  First traversal: split a beam's logits into groups, take each group's max; the
// k-th largest of those maxima (their min when there are exactly k groups) is the R-top-k
// bound, never above the true k-th largest; log_sum_exp in the same pass.  Second
// traversal: keep the logits at or above R-top-k, rescore them as beam_score + logit -
// log_sum_exp, and one sort of that short queue per batch gives the exact top-k.
//
// GB300 design:
//  * One CTA per batch, kFuWarps warps.  The batch's k rows are cut into k * W strips; a warp
//    streams its strip through a ring of kFuRing stages in shared memory, filled by 16-byte
//    asynchronous copies (each lane copies, then reads, its own vectors: no barrier), with
//    kFuRing - 1 stages in flight while one is worked on.  Stages lying wholly inside the row
//    (all but a row's first and last) skip the per-vector range tests and the masking.
//  * First traversal, per stage and in registers: each lane's max of its 64-element block (its
//    8 vectors of the stage) goes to shared memory and into the lane's sorted 8 largest, and
//    a running (max, sum of exp(x - max)) per lane accumulates log_sum_exp.  The blocks
//    partition the row, so the k-th largest block max of a strip is an R-top-k bound for it
//    (groups = blocks: the article's "any split"); at the end of the strip k rounds of a warp
//    max over the lanes' sorted lists give it.
//  * Second traversal: only the blocks whose max reaches the strip's bound (a handful) are
//    read again -- from L2, 128 bytes each -- for their elements x >= bound.  Per row, lse
//    comes from the strips' (max, sum) and R is the largest of the strips' bounds; the
//    candidates at or above R are rescored (beam_score + x - lse, in compensated fp32) into
//    128-bit keys in shared memory and ranked (each key's rank counted against the others;
//    the k of rank < k are the outputs).  Nothing else goes through global memory between
//    the traversals and the rank.
//  * More than kFuList candidates in a strip, more than kFuCap keys (ties), or the forced
//    exact mode send the batch to an exact path: a radix select of every beam's top-k over
//    its logits.
#include <cooperative_groups.h>

#include "ls_device.cuh"
#include "ls_draw.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"
#include "ls_strip.cuh"

namespace lsb {
namespace {

constexpr int kFuWarps = kFuThreads / 32;
constexpr int kFuCap = 512;  // keys the fine rank holds

enum { FROW_LIVE = 0, FROW_FIN = 1, FROW_DEAD = 2 };

// Dynamic shared memory: the per-warp rings of kFuRing stages (the rank keys reuse them once
// the first traversal is done), then the block maxima, [strip][stage of the strip][lane].
constexpr int kFuRing = 3;
constexpr int kFuList = 32;  // candidates a strip keeps
constexpr int kFuHits = 64;  // blocks a strip reads again

struct __align__(16) FuSmem {
  Key* keys;                        // kFuCap keys, over the rings
  float um[kFuWarps], us[kFuWarps];  // strip max and sum of exp(x - max)
  float ur[kFuWarps];                // strip bound: k-th largest block max of the strip
  int ucnt[kFuWarps], uovf[kFuWarps];
  float2 cand[kFuWarps][kFuList];    // the strip's candidates (x, token)
  int hits[kFuWarps][kFuHits];       // the strip's blocks reaching its bound (stage * 32 + lane)
  ScoreBase c[kFuMaxK];  // beam_score - log_sum_exp of each live row
  float beam[kFuMaxK], lse[kFuMaxK], R[kFuMaxK];
  int fin[kFuMaxK], kind[kFuMaxK], ncand[kFuMaxK];
  int nkeys, path;
  // exact path
  unsigned int hist[256];
  unsigned int prefix, pmask;
  int need;
  int wc[kFuWarps];
  // the batch's new parent of each output row (rank order), and each warp's two bulk-copy
  // barriers of the cache refresh
  int opar[kFuMaxK];
  unsigned long long rbar[kFuWarps][2];
  // the one-kernel sampler: each row's top k (best first) and whether it needs the exact path
  float tx[kFuSampRows][kFuMaxK];
  int tv[kFuSampRows][kFuMaxK];
  int spath[kFuSampRows];
  // the cluster step: this CTA's row's top k keys (best first), their count, the row's path,
  // and on the batch's first CTA the gathered rows' offsets and the batch's path
  Key tk[kFuMaxK];
  int ntk, cpath, gpath;
  int goff[kFuMaxK];
};

}  // namespace

size_t beam_fused_smem_bytes(int vpl, int sps) {
  const size_t ring = (size_t)kFuWarps * kFuRing * 32 * vpl * 16;
  return (ring > kFuCap * sizeof(Key) ? ring : kFuCap * sizeof(Key)) + (size_t)kFuWarps * sps * 32 * 4;
}

namespace {

// Append key k (when take) to sm.keys with one shared atomic per warp; returns nothing, the
// count may exceed kFuCap (then the batch takes the exact path).
__device__ __forceinline__ void append_key(FuSmem& sm, bool take, const Key& k) {
  const int lane = threadIdx.x & 31;
  const unsigned m = __ballot_sync(0xffffffffu, take);
  if (m == 0u) return;
  int base = 0;
  if (lane == 0) base = atomicAdd(&sm.nkeys, __popc(m));
  base = __shfl_sync(0xffffffffu, base, 0);
  const int pos = base + __popc(m & ((1u << lane) - 1u));
  if (take && pos < kFuCap) sm.keys[pos] = k;
}

// Rank of every key among the keys; ranks 0..K-1 are written as the batch's outputs.
__device__ void rank_and_write(const StepParams& p, FuSmem& sm, int b) {
  const int n = sm.nkeys < kFuCap ? sm.nkeys : kFuCap;
  const int K = p.k;
  for (int i = threadIdx.x; i < n; i += kFuThreads) {
    const Key ki = sm.keys[i];
    int r0 = 0, r1 = 0, q = 0;
#pragma unroll 1
    for (; q + 1 < n; q += 2) {
      r0 += key_less(sm.keys[q], ki);
      r1 += key_less(sm.keys[q + 1], ki);
    }
    if (q < n) r0 += key_less(sm.keys[q], ki);
    const int rank = r0 + r1;
    if (rank < K) {
      const int o = b * K + rank;
      const int parent = key_parent(ki), token = key_token(ki);
      sm.opar[rank] = parent;
      p.out_token[o] = token;
      p.out_parent[o] = parent;
      p.out_score[o] = key_score(ki);
      if (p.out_finished) p.out_finished[o] = (sm.fin[parent] || token == p.eos) ? 1 : 0;
    }
  }
}

// Exact top-K of live row j by (x descending, token ascending): a radix select of the K-th
// order key over the row's logits, 8 bits a pass, then the elements above it and the first
// `need` equal to it in token order.  All threads call it.
template <int DT, bool BIAS>
__device__ void exact_row(const StepParams& p, FuSmem& sm, long long row, int j) {
  constexpr int ES = Traits<DT>::kBytes;
  const int K = p.k, V = p.vocab;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned char* rowp = static_cast<const unsigned char*>(p.logits) + (size_t)row * V * ES;
  auto xat = [&](int i) -> float {
    float x = load_elem<DT>(rowp + (size_t)i * ES);
    if constexpr (BIAS) x += __ldg(p.bias + i);
    return x;
  };
  if (tid == 0) {
    sm.prefix = 0;
    sm.pmask = 0;
    sm.need = K;
  }
  __syncthreads();
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kFuThreads) sm.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sm.prefix, pmask = sm.pmask;
    for (int i = tid; i < V; i += kFuThreads) {
      const uint32_t o = float_ord(xat(i));
      if ((o & pmask) == prefix) atomicAdd(&sm.hist[(o >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      const int need = sm.need;
      unsigned int cum = 0;
      int dgt = 255;
      for (; dgt > 0; --dgt) {
        if (cum + sm.hist[dgt] >= (unsigned)need) break;
        cum += sm.hist[dgt];
      }
      sm.need = need - (int)cum;
      sm.prefix = prefix | ((uint32_t)dgt << shift);
      sm.pmask = pmask | (255u << shift);
    }
    __syncthreads();
  }
  const uint32_t tkey = sm.prefix;
  const int need_eq = sm.need;
  const ScoreBase c = sm.c[j];
  for (int base = 0; base < V; base += kFuThreads) {
    const int i = base + tid;
    float x = 0.0f;
    bool take = false;
    if (i < V) {
      x = xat(i);
      take = float_ord(x) > tkey;
    }
    append_key(sm, take, make_key(score_of(c, x), j, x, i));
  }
  __syncthreads();
  // the first need_eq elements equal to the K-th key, in token order
  int taken = 0;
  for (int base = 0; base < V && taken < need_eq; base += kFuThreads) {
    const int i = base + tid;
    float x = 0.0f;
    bool eq = false;
    if (i < V) {
      x = xat(i);
      eq = float_ord(x) == tkey;
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) sm.wc[warp] = __popc(ballot);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kFuWarps; ++w) {
      before += (w < warp) ? sm.wc[w] : 0;
      total += sm.wc[w];
    }
    const int off = taken + before + __popc(ballot & ((1u << lane) - 1u));
    append_key(sm, eq && off < need_eq, make_key(score_of(c, x), j, x, i));
    taken += total;
    __syncthreads();
  }
  __syncthreads();
}

// The in-place cache refresh of batch b by the parents in sm.opar, after the step: the
// warps take the batch's items (layer, heads [h0, h0 + rf_hg), one tile of their slabs) in
// turn, and lane 0 of each runs a two-buffer pipeline in the warp's part of the rings, as the
// standalone bulk-copy refresh does: the bulk loads of the slabs item i needs are issued
// before the bulk stores of item i-1's changed rows, and a buffer is refilled only after the
// stores that read it.  Every row reads the state before the step: an item's stores start
// only once all of its loads have landed, and items touch disjoint bytes.  Waits are bounded;
// one that runs out sets the timeout bit and lets the copies in flight land.
__device__ void refresh_batch(const StepParams& p, FuSmem& sm, unsigned char* wbuf, uint32_t buf_bytes, int b) {
  const int K = p.k, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned changed = 0u, needed = 0u;
  for (int j = 0; j < K; ++j) {
    const int q = sm.opar[j];
    if (q != j) {
      changed |= 1u << j;
      needed |= 1u << q;
    }
  }
  if (changed == 0u || lane != 0) return;
  const int HG = p.rf_hg, TB = p.rf_tile;
  const long long groups = (p.rf_heads + HG - 1) / HG;
  const long long ntiles = (p.rf_slab_bytes + TB - 1) / TB;
  const long long nitems = (long long)p.rf_layers * groups * ntiles;
  const uint32_t bar0 = smem_addr(&sm.rbar[warp][0]), bar1 = smem_addr(&sm.rbar[warp][1]);
  uint32_t uses0 = 0u, uses1 = 0u;  // completed-or-pending fills of each buffer
  int cur = 0;
  bool aborted = false, have_prev = false;
  unsigned char* pv_base = nullptr;
  int pv_tb = 0, pv_hg = 0, pv_buf = 0;
  uint32_t pv_parity = 0;
  auto finish_prev = [&]() {
    if (!mbar_wait_bounded(pv_buf ? bar1 : bar0, pv_parity, p.spin_limit_ns)) {
      aborted = true;
      return;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const unsigned char* src = wbuf + (size_t)pv_buf * buf_bytes;
    for (int j = 0; j < K; ++j) {
      if (!((changed >> j) & 1u)) continue;
      const int slot = __popc(needed & ((1u << sm.opar[j]) - 1u));
      for (int hh = 0; hh < pv_hg; ++hh)
        bulk_store(pv_base + (size_t)j * p.rf_row_stride + (size_t)hh * p.rf_slab_stride,
                   smem_addr(src + ((size_t)slot * pv_hg + hh) * pv_tb), (uint32_t)pv_tb);
    }
    bulk_commit();
  };
  const int nneed = __popc(needed);
  for (long long it = warp; it < nitems && !aborted; it += kFuWarps) {
    const long long unit = it / ntiles;
    const long long tile = it - unit * ntiles;
    const int l = (int)(unit / groups);
    const int h0 = (int)(unit - (long long)l * groups) * HG;
    const int hg = min(HG, p.rf_heads - h0);
    const long long t0 = tile * TB;
    const int tb = (int)min((long long)TB, p.rf_slab_bytes - t0);
    unsigned char* base = p.rf_cache + (size_t)l * p.rf_layer_stride + (size_t)b * K * p.rf_row_stride +
                          (size_t)h0 * p.rf_slab_stride + t0;
    bulk_wait_read<0>();  // buffer `cur` was last read by the stores of the item before the previous one
    const uint32_t bcur = cur ? bar1 : bar0;
    mbar_arrive_expect_tx(bcur, (uint32_t)(nneed * hg * tb));
    unsigned char* dst = wbuf + (size_t)cur * buf_bytes;
    int slot = 0;
    for (int q = 0; q < K; ++q) {
      if (!((needed >> q) & 1u)) continue;
      for (int hh = 0; hh < hg; ++hh)
        bulk_load_plain(smem_addr(dst + ((size_t)slot * hg + hh) * tb),
                        base + (size_t)q * p.rf_row_stride + (size_t)hh * p.rf_slab_stride, (uint32_t)tb, bcur);
      ++slot;
    }
    if (have_prev) finish_prev();
    have_prev = true;
    pv_base = base;
    pv_tb = tb;
    pv_hg = hg;
    pv_buf = cur;
    uint32_t& uses = cur ? uses1 : uses0;
    pv_parity = uses & 1u;
    ++uses;
    cur ^= 1;
  }
  if (have_prev && !aborted) finish_prev();
  if (aborted) {
    atomicOr(p.status, kDevTimeout);
    if (uses0 > 0) mbar_wait_bounded(bar0, (uses0 - 1) & 1u, 2000000000LL);
    if (uses1 > 0) mbar_wait_bounded(bar1, (uses1 - 1) & 1u, 2000000000LL);
  }
  bulk_wait_all();
}

// Modes of the kernel: the batch step (one CTA per batch), the sampler (kFuSampRows rows per
// CTA), and the cluster step (one CTA per row, a batch's k CTAs a thread-block cluster).
enum { kModeBatch = 0, kModeSample = 1, kModeCluster = 2 };

template <int DT, bool BIAS, int VPL, int MODE>
__global__ void __launch_bounds__(kFuThreads, 2) beam_fused_kernel(const StepParams p) {
  constexpr bool SAMP = MODE == kModeSample;
  constexpr bool CL = MODE == kModeCluster;
  constexpr int VEC = Traits<DT>::kVec;
  constexpr int ES = Traits<DT>::kBytes;
  constexpr int CV = 32 * VPL;                       // vectors per stage
  constexpr bool kPacked = (DT != DT_F32) && !BIAS;  // the block max on packed 16-bit pairs
  constexpr int EL = VPL * VEC;                      // elements per lane per stage (one block)
  __shared__ FuSmem sm;
  extern __shared__ __align__(128) unsigned char fu_dyn[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.k, V = p.vocab, W = p.nc;  // W strips per row, one warp per strip
  // rows per CTA: the batch's k beams, kFuSampRows independent rows for the sampler, or one
  // beam of the batch in the cluster step (its rank in the cluster)
  const int NR = SAMP ? kFuSampRows : (CL ? 1 : K);
  const int crank = CL ? (int)cooperative_groups::this_cluster().block_rank() : 0;
  const int b = CL ? (int)blockIdx.x / K : (int)blockIdx.x;  // the batch (the row group when SAMP)
  const int jb = CL ? crank : 0;                            // the batch row of this CTA's first row
  const int SPS = p.stages;                  // block-max rows kept per strip
  unsigned char* ring = fu_dyn + (size_t)warp * kFuRing * CV * 16;
  float* bmax = reinterpret_cast<float*>(fu_dyn + (size_t)kFuWarps * kFuRing * CV * 16);
  const int row_bytes = V * ES;
  const unsigned char* logits = static_cast<const unsigned char*>(p.logits);

  // inputs may come from the previous kernel of the stream
  grid_dependency_wait();
  if constexpr (SAMP) {
    if (tid < NR) {
      sm.beam[tid] = 0.0f;
      sm.fin[tid] = (long long)b * NR + tid >= p.rows ? 1 : 0;  // past the last row: skipped
      sm.ncand[tid] = 0;
      sm.spath[tid] = 0;
    }
  } else if (tid < K) {
    sm.beam[tid] = p.beam[b * K + tid];
    sm.fin[tid] = (p.finished && p.finished[b * K + tid]) ? 1 : 0;
    sm.ncand[tid] = 0;
  }
  if (tid == 0) {
    sm.keys = reinterpret_cast<Key*>(fu_dyn);
    sm.nkeys = 0;
    sm.path = (p.flags & kFlagForceExact) ? 2 : 0;
  }
  if (p.rf_cache && tid == 0) {
    for (int w = 0; w < kFuWarps; ++w) {
      mbar_init(smem_addr(&sm.rbar[w][0]), 1);
      mbar_init(smem_addr(&sm.rbar[w][1]), 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // Geometry of row j (the row's index in the batch, or in the CTA's group for the sampler):
  // 16-byte aligned vectors covering it, stages of CV vectors.
  struct RowGeo {
    const uint4* rb;  // first vector (16-byte aligned, may start before the row)
    int lead;         // bytes of that vector before the row
    int nv, ns;
  };
  auto geo = [&](int j) -> RowGeo {
    RowGeo g;
    const unsigned char* rowp = logits + (SAMP ? (size_t)b * NR + j : (size_t)b * K + j) * row_bytes;
    g.lead = (int)(reinterpret_cast<uintptr_t>(rowp) & 15);
    g.rb = reinterpret_cast<const uint4*>(rowp - g.lead);
    g.nv = (g.lead + row_bytes + 15) >> 4;
    g.ns = (g.nv + CV - 1) / CV;
    return g;
  };
  // Block (stage q, lane l) of the row: vectors q * CV + l + 32 r, r < VPL; elements outside
  // the row read as -inf.
  auto load_block = [&](const RowGeo& g, uint4 (&d)[VPL], int q, int l) {
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      const int jv = q * CV + l + 32 * r;
      const uint32_t w = Traits<DT>::kNegInfWord;
      d[r] = jv < g.nv ? __ldcs(g.rb + jv) : make_uint4(w, w, w, w);
    }
  };
  auto mask_block = [&](const RowGeo& g, uint4 (&d)[VPL], int q, int l) {
    const int j0 = q * CV;
    if (j0 * 16 - g.lead >= 0 && (j0 + CV) * 16 - g.lead <= row_bytes) return;  // interior stage
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      const int base_b = (j0 + l + 32 * r) * 16 - g.lead;  // row byte offset of element 0
      if (base_b < 0 || base_b + 16 > row_bytes) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const int eb = base_b + e * ES;
          if (eb < 0 || eb >= row_bytes) set_neg_inf<DT>(d[r], e);
        }
      }
    }
  };
  // x = logit + bias of the block as floats (bias and f32 variants)
  auto block_x = [&](const RowGeo& g, const uint4 (&d)[VPL], int q, int l, float (&xf)[EL]) {
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      float x[VEC];
      unpack<DT>(d[r], x);
      if constexpr (BIAS) {
        const int base_b = (q * CV + l + 32 * r) * 16 - g.lead;
        const int v0 = base_b / ES;
        if (base_b >= 0 && base_b + 16 <= row_bytes && ((reinterpret_cast<uintptr_t>(p.bias + v0) & 15) == 0)) {
#pragma unroll
          for (int e = 0; e < VEC; e += 4) {
            const float4 bb = __ldg(reinterpret_cast<const float4*>(p.bias + v0 + e));
            x[e] += bb.x;
            x[e + 1] += bb.y;
            x[e + 2] += bb.z;
            x[e + 3] += bb.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const int eb = base_b + e * ES;
            if (eb >= 0 && eb < row_bytes) x[e] += __ldg(p.bias + eb / ES);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) xf[r * VEC + e] = x[e];
    }
  };

  // ---------------------------------------------------------------- first traversal
  // warp u streams strip s = u mod W of row j = u / W: stages s, s + W, ...
  const int nunits = NR * W;
  if (warp < nunits) {
    const int u = warp, j = u / W + jb, s = u - (j - jb) * W;  // j: the row's index in the batch
    float ml = -INFINITY;  // lane's running max
    float cl = 0.0f;       // the lane's sum is sl = sum of 2^(x log2e + cl), cl = -ml log2e rounded
    float sl = 0.0f;
    float t[8];  // the lane's 8 largest block maxima, descending (insertion as the stages stream)
#pragma unroll
    for (int i8 = 0; i8 < 8; ++i8) t[i8] = -INFINITY;
    if (!sm.fin[j]) {
      const RowGeo g = geo(j);
      // the strip's stages go through a ring of kFuRing stage buffers in shared memory,
      // filled by 16-byte asynchronous copies (each lane copies, then reads, its own
      // vectors: no barrier), kFuRing - 1 stages in flight while one is worked on.  A stage
      // whose vectors all lie inside the row (every one but a row's first and last) takes
      // the short path: no per-vector range test, no masking.
      const uint64_t pol = l2_evict_first_policy();
      const int in_lo = (g.lead + CV * 16 - 1) / (CV * 16);     // first stage starting inside the row
      const int in_hi = (g.lead + row_bytes) / (CV * 16) - 1;  // last stage ending inside the row
      auto issue = [&](int q, int slot) {
        unsigned char* dst = ring + (slot * VPL * 32 + lane) * 16;
        const uint4* src = g.rb + q * CV + lane;
        if (q >= in_lo && q <= in_hi) {
#pragma unroll
          for (int r = 0; r < VPL; ++r) cp_async16(smem_addr(dst + r * 512), src + 32 * r, pol);
        } else if (q < g.ns) {
#pragma unroll
          for (int r = 0; r < VPL; ++r) {
            const int jv = q * CV + lane + 32 * r;
            if (jv < g.nv) cp_async16(smem_addr(dst + r * 512), src + 32 * r, pol);
          }
        }
        cp_async_commit();
      };
      uint4 d[VPL];
      int q = s, i = 0;
#pragma unroll
      for (int a = 0; a < kFuRing - 1; ++a) issue(q + a * W, a);
      int slot = 0, islot = kFuRing - 1;  // the stage worked on, the stage being issued
#pragma unroll 1
      for (; q < g.ns; q += W, ++i) {
        cp_async_wait<kFuRing - 2>();
        const unsigned char* src = ring + (slot * VPL * 32 + lane) * 16;
        const bool inner = q >= in_lo && q <= in_hi;
        if (inner) {
#pragma unroll
          for (int r = 0; r < VPL; ++r) d[r] = *reinterpret_cast<const uint4*>(src + r * 512);
        } else {
#pragma unroll
          for (int r = 0; r < VPL; ++r) {
            const int jv = q * CV + lane + 32 * r;
            const uint32_t w = Traits<DT>::kNegInfWord;
            d[r] = jv < g.nv ? *reinterpret_cast<const uint4*>(src + r * 512) : make_uint4(w, w, w, w);
          }
        }
        issue(q + (kFuRing - 1) * W, islot);
        slot = slot == kFuRing - 1 ? 0 : slot + 1;
        islot = islot == kFuRing - 1 ? 0 : islot + 1;
        if (!inner) mask_block(g, d, q, lane);
        float xf[kPacked ? 1 : EL];
        if constexpr (!kPacked) block_x(g, d, q, lane, xf);
        // the block max
        float lm;
        if constexpr (kPacked) {
          uint32_t t = hmax2_bits<DT>(hmax2_bits<DT>(d[0].x, d[0].y), hmax2_bits<DT>(d[0].z, d[0].w));
#pragma unroll
          for (int r = 1; r < VPL; ++r)
            t = hmax2_bits<DT>(t, hmax2_bits<DT>(hmax2_bits<DT>(d[r].x, d[r].y), hmax2_bits<DT>(d[r].z, d[r].w)));
          lm = hpair_max<DT>(t);
        } else {
          lm = xf[0];
#pragma unroll
          for (int q2 = 1; q2 < EL; ++q2) lm = fmaxf(lm, xf[q2]);
        }
        bmax[(u * SPS + i) * 32 + lane] = lm;
        if (lm > t[7]) {
          float v = lm;
#pragma unroll
          for (int q2 = 0; q2 < 8; ++q2) {  // insert, keeping t descending
            const float hi = fmaxf(t[q2], v);
            v = fminf(t[q2], v);
            t[q2] = hi;
          }
        }
        // log_sum_exp: the lane's sum is kept as sum of 2^(x log2e + c) with c = -max log2e
        // rounded (one fused multiply-add per term); rescaled by 2^(c_new - c_old) when the
        // lane's max rises, and corrected for the rounding of c once, at the end of the strip
        const float mn = fmaxf(ml, lm);
        const float cn = mn == -INFINITY ? 0.0f : -mn * kLog2e;
        sl = ml == -INFINITY ? 0.0f : sl * fast_exp2(cn - cl);
        cl = cn;
        ml = mn;
        const float2 L2 = make_float2(kLog2e, kLog2e), c2 = make_float2(cn, cn);
        float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
        auto term2 = [&](float2 x) {
          const float2 t = __ffma2_rn(x, L2, c2);
          return make_float2(fast_exp2(t.x), fast_exp2(t.y));
        };
        if constexpr (kPacked) {
#pragma unroll
          for (int r = 0; r < VPL; ++r) {
            const uint32_t w[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              float2 f0, f1;
              if constexpr (DT == DT_F16) {
                f0 = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                f1 = __half22float2(*reinterpret_cast<const __half2*>(&w[e + 1]));
              } else {
                f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
                f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e + 1]));
              }
              a0 = __fadd2_rn(a0, term2(f0));
              a1 = __fadd2_rn(a1, term2(f1));
            }
          }
        } else {
#pragma unroll
          for (int q2 = 0; q2 < EL; q2 += 4) {
            a0 = __fadd2_rn(a0, term2(make_float2(xf[q2], xf[q2 + 1])));
            a1 = __fadd2_rn(a1, term2(make_float2(xf[q2 + 2], xf[q2 + 3])));
          }
        }
        const float2 a = __fadd2_rn(a0, a1);
        sl += a.x + a.y;
      }
      cp_async_wait<0>();  // the ring becomes the key array: no copy may still land in it
    }
    // end of the strip: the lanes' (max, sum) merged
    float M = ml;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // sl * 2^(-(ml log2e + cl)) is the lane's sum of exp(x - ml); then rescaled to M
    float S = (ml == -INFINITY) ? 0.0f : sl * fast_exp2(-fmaf(ml, kLog2e, cl) + (ml - M) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);

    // the strip's bound: the k-th largest of its block maxima (each lane has kept the 8
    // largest of its own blocks; k rounds of a warp max take them out in order)
    const RowGeo g = geo(j);
    const int nst = (!sm.fin[j] && s < g.ns) ? (g.ns - s + W - 1) / W : 0;
    float Rs = -INFINITY;
    for (int r = 0; r < K; ++r) {
      float m = t[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const unsigned who = __ballot_sync(0xffffffffu, t[0] == m);
      if (lane == __ffs(who) - 1) {
#pragma unroll
        for (int q2 = 0; q2 < 7; ++q2) t[q2] = t[q2 + 1];
        t[7] = -INFINITY;
      }
      Rs = m;
    }
    // second traversal of the strip: its blocks whose max reaches the bound are read again,
    // all at once (lane h takes hit h), and their elements x >= bound kept as candidates
    const float thr = fmaxf(Rs, lowest_finite<DT>());  // -inf elements are never candidates
    int nh = 0;
    for (int i = 0; i < nst; ++i) {
      const bool hit = bmax[(u * SPS + i) * 32 + lane] >= thr;
      const unsigned hm = __ballot_sync(0xffffffffu, hit);
      const int pos = nh + __popc(hm & ((1u << lane) - 1u));
      if (hit && pos < kFuHits) sm.hits[u][pos] = i * 32 + lane;
      nh += __popc(hm);
    }
    bool ovf = nh > kFuHits;
    if (lane == 0) sm.ucnt[u] = 0;
    __syncwarp();
    for (int h0 = 0; h0 < nh && !ovf; h0 += 32) {
      const int h = h0 + lane;
      if (h < nh) {
        const int i = sm.hits[u][h] >> 5, l = sm.hits[u][h] & 31;
        const int q = s + i * W;
        uint4 d[VPL];
        load_block(g, d, q, l);
        mask_block(g, d, q, l);
        float xf[kPacked ? 1 : EL];
        if constexpr (!kPacked) block_x(g, d, q, l, xf);
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
          uint32_t m;
          if constexpr (kPacked) {
            m = hvec_ge_mask<DT>(d[r], thr);
          } else {
            m = 0;
#pragma unroll
            for (int e = 0; e < VEC; ++e) m |= (xf[r * VEC + e] >= thr ? 1u : 0u) << e;
          }
          while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1;
            float x;
            if constexpr (kPacked) {
              x = vec_elem_f<DT>(d[r], e);
            } else {
              float tv = xf[r * VEC];
#pragma unroll
              for (int q2 = 1; q2 < VEC; ++q2) tv = q2 == e ? xf[r * VEC + q2] : tv;
              x = tv;
            }
            const int v = ((q * CV + l + 32 * r) * 16 - g.lead) / ES + e;
            const int pos = atomicAdd(&sm.ucnt[u], 1);
            if (pos < kFuList) sm.cand[u][pos] = make_float2(x, __int_as_float(v));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      sm.um[u] = M;
      sm.us[u] = S;
      sm.ur[u] = Rs;
      sm.uovf[u] = (ovf || sm.ucnt[u] > kFuList) ? 1 : 0;
    }
  }
  __syncthreads();

  if constexpr (SAMP) {
    // ---------------------------------------------------------------- per row: the draw
    // warp j takes row j: lse from its strips' (max, sum), R = the largest strip bound, the
    // row's candidates at or above R ranked (larger x, then smaller token) into its top k,
    // and the draw at u[row]
    if (warp < NR && !sm.fin[warp]) {
      const int j = warp, u0 = j * W;
      const long long row = (long long)b * NR + j;
      const float mu = lane < W ? sm.um[u0 + lane] : -INFINITY;
      float M = mu;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float S = (lane < W && mu != -INFINITY) ? sm.us[u0 + lane] * exp2f((mu - M) * kLog2e) : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      float Rr = lane < W ? sm.ur[u0 + lane] : -INFINITY;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Rr = fmaxf(Rr, __shfl_xor_sync(0xffffffffu, Rr, o));
      const bool ovf = __any_sync(0xffffffffu, lane < W && sm.uovf[u0 + lane] != 0);
      const float lse = M == -INFINITY ? -INFINITY : __fadd_rn(M, logf(S));
      // candidate `lane` of each strip of the row, kept when at or above R
      float cx[kFuWarps / kFuSampRows];
      int cv[kFuWarps / kFuSampRows];
      bool ck[kFuWarps / kFuSampRows];
      int ntot = 0;
#pragma unroll
      for (int t = 0; t < kFuWarps / kFuSampRows; ++t) {
        const int n = t < W ? min(sm.ucnt[u0 + t], kFuList) : 0;
        const float2 en = lane < n ? sm.cand[u0 + t][lane] : make_float2(-INFINITY, 0.0f);
        ck[t] = lane < n && en.x >= Rr;
        cx[t] = en.x;
        cv[t] = __float_as_int(en.y);
        ntot += __popc(__ballot_sync(0xffffffffu, ck[t]));
      }
      const bool forced = (p.flags & kFlagForceExact) != 0;
      const bool exact = forced || ovf || ntot < K;
      if (!exact) {
#pragma unroll
        for (int t = 0; t < kFuWarps / kFuSampRows; ++t) {
          if (ck[t]) {
            int rank = 0;
            for (int t2 = 0; t2 < W; ++t2) {
              const int n2 = min(sm.ucnt[u0 + t2], kFuList);
              for (int i = 0; i < n2; ++i) {
                const float2 e = sm.cand[u0 + t2][i];
                const int ev = __float_as_int(e.y);
                rank += (e.x >= Rr) & ((e.x > cx[t]) | ((e.x == cx[t]) & (ev < cv[t])));
              }
            }
            if (rank < K) {
              sm.tx[j][rank] = cx[t];
              sm.tv[j][rank] = cv[t];
            }
          }
        }
        __syncwarp();
        draw_topk(sm.tx[j], sm.tv[j], K, p.top_p, lse, p.u[row], (int)row, p.out_token, p.out_logprob);
      }
      if (lane == 0) {
        sm.spath[j] = exact ? 1 : 0;
        sm.lse[j] = lse;
        RowStat st;
        st.lse = lse;
        st.rtopk = Rr;
        st.ncand = exact ? -1 : ntot;
        st.pad = 0;
        p.rowstat[row] = st;
        p.bstat[row] = forced ? 2 : (exact ? 1 : 0);
      }
    }
    __syncthreads();
    // a row that lost a candidate, or holds fewer than k at or above R: its exact top k by a
    // radix select over the row (the whole CTA), ranked by x (the keys' score is x here), then
    // the draw
    for (int j = 0; j < NR; ++j) {
      if (!sm.spath[j] || sm.fin[j]) continue;  // CTA-uniform
      if (tid == 0) {
        sm.nkeys = 0;
        sm.c[j] = ScoreBase{0.0f, 0.0f};
      }
      __syncthreads();
      const long long row = (long long)b * NR + j;
      exact_row<DT, BIAS>(p, sm, row, j);
      if (warp == 0) {
        const int n = min(sm.nkeys, kFuCap);
        for (int i = lane; i < n; i += 32) {
          const Key ki = sm.keys[i];
          int rank = 0;
          for (int q = 0; q < n; ++q) rank += key_less(sm.keys[q], ki);
          if (rank < K) {
            sm.tx[j][rank] = key_score(ki);
            sm.tv[j][rank] = key_token(ki);
          }
        }
        __syncwarp();
        draw_topk(sm.tx[j], sm.tv[j], K, p.top_p, sm.lse[j], p.u[row], (int)row, p.out_token, p.out_logprob);
      }
      __syncthreads();
    }
    return;
  }

  // ---------------------------------------------------------------- per row: lse, R, keys
  // warp j merges row j's strips -- lse from their (max, sum), R = the largest of their
  // bounds (each is at most the row's k-th largest) -- and appends the row's keys: the strips'
  // candidates at or above R, rescored as beam_score + x - lse; a finished beam offers
  // (eos_id, beam score), a beam with no finite score k tokens
  if (warp < NR) {
    const int j = jb + warp, u0 = warp * W;  // j: the row's index in the batch
    const float mu = lane < W ? sm.um[u0 + lane] : -INFINITY;
    float M = mu;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = (lane < W && mu != -INFINITY) ? sm.us[u0 + lane] * exp2f((mu - M) * kLog2e) : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    float Rr = lane < W ? sm.ur[u0 + lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Rr = fmaxf(Rr, __shfl_xor_sync(0xffffffffu, Rr, o));
    const bool ovf = __any_sync(0xffffffffu, lane < W && sm.uovf[u0 + lane] != 0);
    const float beam = sm.beam[j];
    const int kind = sm.fin[j] ? FROW_FIN : ((M == -INFINITY || beam == -INFINITY) ? FROW_DEAD : FROW_LIVE);
    const float log_s = logf(S);
    const ScoreBase c = kind == FROW_LIVE ? score_base(beam, M, log_s) : ScoreBase{0.0f, 0.0f};
    if (lane == 0) {
      sm.kind[j] = kind;
      sm.R[j] = Rr;
      sm.lse[j] = kind == FROW_FIN ? __int_as_float(0x7fc00000) : (M == -INFINITY ? -INFINITY : __fadd_rn(M, log_s));
      sm.c[j] = c;
      if (ovf && kind == FROW_LIVE) atomicMax(&sm.path, 1);
    }
    int nc = 0;
    if (kind == FROW_LIVE) {
      if (!ovf) {
        for (int t = 0; t < W; ++t) {
          const int u = u0 + t;
          const int n = min(sm.ucnt[u], kFuList);
          float2 en = make_float2(0.0f, 0.0f);
          if (lane < n) en = sm.cand[u][lane];
          const bool take = lane < n && en.x >= Rr;
          append_key(sm, take, make_key(score_of(c, en.x), j, en.x, __float_as_int(en.y)));
          nc += __popc(__ballot_sync(0xffffffffu, take));
        }
      }
    } else {
      const bool take = kind == FROW_DEAD ? lane < K : lane == 0;
      append_key(sm, take, kind == FROW_FIN ? make_key(beam, j, 0.0f, p.eos) : make_key(-INFINITY, j, 0.0f, lane));
      nc = kind == FROW_FIN ? 1 : K;
    }
    if (lane == 0) sm.ncand[j] = nc;
  }
  __syncthreads();
  // any strip that lost a candidate, or more keys than the rank holds: the exact path
  const int path = sm.path != 0 ? sm.path : (sm.nkeys > kFuCap ? 3 : 0);
  if (path != 0) {
    // exact path: every live beam's top-K by radix select over its logits (the barrier first:
    // every thread has read the key count that chose the path)
    __syncthreads();
    if (tid == 0) sm.nkeys = 0;
    __syncthreads();
    for (int jl = 0; jl < NR; ++jl) {
      const int j = jb + jl;
      const int kind = sm.kind[j];
      if (kind == FROW_LIVE) {
        exact_row<DT, BIAS>(p, sm, (long long)b * K + j, j);
      } else {
        if (tid < K && (kind == FROW_DEAD || tid == 0)) {
          const int pos = atomicAdd(&sm.nkeys, 1);
          sm.keys[pos] = kind == FROW_FIN ? make_key(sm.beam[j], j, 0.0f, p.eos) : make_key(-INFINITY, j, 0.0f, tid);
        }
        __syncthreads();
      }
    }
  }
  if constexpr (CL) {
    // this row's top k keys, best first (the batch's top k holds no other key of the row)
    const int n = min(sm.nkeys, kFuCap);
    for (int i = tid; i < n; i += kFuThreads) {
      const Key ki = sm.keys[i];
      int r0 = 0;
      for (int q = 0; q < n; ++q) r0 += key_less(sm.keys[q], ki);
      if (r0 < K) sm.tk[r0] = ki;
    }
    if (tid == 0) {
      sm.ntk = min(n, K);
      sm.cpath = path;
    }
    cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
    cl.sync();  // every row of the batch has its top k
    if (crank == 0) {
      // the batch's first CTA gathers the rows' top k (distributed shared memory) and ranks them
      if (tid == 0) {
        int off = 0, pm = 0;
        for (int r = 0; r < K; ++r) {
          const FuSmem* ps = cl.map_shared_rank(&sm, (unsigned)r);
          sm.goff[r] = off;
          off += ps->ntk;
          pm = max(pm, ps->cpath);
        }
        sm.nkeys = off;
        sm.gpath = pm;
      }
      __syncthreads();
      for (int idx = tid; idx < K * K; idx += kFuThreads) {
        const int r = idx / K, i = idx - r * K;
        const FuSmem* ps = cl.map_shared_rank(&sm, (unsigned)r);
        if (i < ps->ntk) sm.keys[sm.goff[r] + i] = ps->tk[i];
      }
      __syncthreads();
      rank_and_write(p, sm, b);
      if (tid == 0) p.bstat[b] = sm.gpath;
    }
    cl.sync();  // a row's shared memory stays until the gather has read it
  } else {
    rank_and_write(p, sm, b);
    if (tid == 0) p.bstat[b] = path;
  }
  if (tid < NR) {
    const int j = jb + tid;
    RowStat st;
    st.lse = sm.lse[j];
    st.rtopk = sm.R[j];
    st.ncand = path != 0 ? -1 : sm.ncand[j];
    st.pad = 0;
    p.rowstat[b * K + j] = st;
  }
  if (!CL && p.rf_cache) {
    // every thread's reads of the keys and the rings are done before they become buffers of
    // bulk copies (the async proxy)
    __syncthreads();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t wbytes = (uint32_t)(kFuRing * CV * 16);
    refresh_batch(p, sm, fu_dyn + (size_t)warp * wbytes, wbytes / 2, b);
  }
}

template <int DT, bool BIAS, int VPL, int MODE>
cudaError_t launch_t(const StepParams& p, cudaStream_t stream) {
  const unsigned grid = MODE == kModeSample    ? (unsigned)((p.rows + kFuSampRows - 1) / kFuSampRows)
                        : MODE == kModeCluster ? (unsigned)p.batch * (unsigned)p.k
                                               : (unsigned)p.batch;
  PdlLaunch l(dim3(grid), dim3(kFuThreads), beam_fused_smem_bytes(VPL, p.stages), stream);
  cudaLaunchAttribute attr[2];
  if (MODE == kModeCluster) {
    // a batch's k CTAs form one cluster (k a power of two up to 8)
    attr[0] = l.attr[0];
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.k;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    l.cfg.attrs = attr;
    l.cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&l.cfg, beam_fused_kernel<DT, BIAS, VPL, MODE>, p);
}

template <int DT, bool BIAS, int VPL>
cudaError_t config_t() {
  const int smem = (int)beam_fused_smem_bytes(VPL, kFuMaxStages);
  cudaError_t e = cudaFuncSetAttribute(beam_fused_kernel<DT, BIAS, VPL, kModeBatch>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(beam_fused_kernel<DT, BIAS, VPL, kModeSample>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(beam_fused_kernel<DT, BIAS, VPL, kModeCluster>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

}  // namespace

cudaError_t beam_fused_config() {
  cudaError_t e = config_t<DT_F32, false, 4>();
  if (e == cudaSuccess) e = config_t<DT_F32, true, 4>();
  if (e == cudaSuccess) e = config_t<DT_F16, false, 8>();
  if (e == cudaSuccess) e = config_t<DT_F16, true, 4>();
  if (e == cudaSuccess) e = config_t<DT_BF16, false, 8>();
  if (e == cudaSuccess) e = config_t<DT_BF16, true, 4>();
  return e;
}

int beam_fused_refresh_buffer(int dtype, bool bias) {
  const int vpl = (dtype == DT_F32 || bias) ? 4 : 8;  // as launch_beam_fused picks it
  return kFuRing * 32 * vpl * 16 / 2;
}

template <int MODE>
cudaError_t launch_any(const StepParams& p, int dtype, cudaStream_t stream) {
  const bool bias = p.bias != nullptr;
  switch (dtype) {
    case DT_F32:
      return bias ? launch_t<DT_F32, true, 4, MODE>(p, stream) : launch_t<DT_F32, false, 4, MODE>(p, stream);
    case DT_F16:
      return bias ? launch_t<DT_F16, true, 4, MODE>(p, stream) : launch_t<DT_F16, false, 8, MODE>(p, stream);
    case DT_BF16:
      return bias ? launch_t<DT_BF16, true, 4, MODE>(p, stream) : launch_t<DT_BF16, false, 8, MODE>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_beam_fused(const StepParams& p, int dtype, cudaStream_t stream) {
  return launch_any<kModeBatch>(p, dtype, stream);
}

cudaError_t launch_sample_fused(const StepParams& p, int dtype, cudaStream_t stream) {
  return launch_any<kModeSample>(p, dtype, stream);
}

cudaError_t launch_beam_cluster(const StepParams& p, int dtype, cudaStream_t stream) {
  return launch_any<kModeCluster>(p, dtype, stream);
}

}  // namespace lsb
