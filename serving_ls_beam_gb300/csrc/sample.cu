// Sampling kernel K5: the draw of one token per sequence from the top-k (optionally
// top-p) candidates of its logits, after K1 has streamed every row once.  This two-kernel
// sampler serves top_k > 8 and row counts too small to fill the GPU; otherwise the one-kernel
// sampler in beam_fused.cu runs.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), decoding section: besides
// beam search, decoding by sampling.  The hierarchical first traversal applies unchanged:
// K1 gives per chunk (max, sum of exp, group maxima) and the chunk's survivors above its
// R-top-k bound; this kernel merges them into the row's log_sum_exp and R-top-k, keeps the
// survivors above that bound, takes the exact top-k among them, and draws by inverse CDF
// at the caller's uniform u.
//
// GB300 design: one warp per row, eight rows per CTA, launched with programmatic
// dependent launch behind K1.  A warp merges its row's chunk records (group maxima through
// shared-memory atomics on order-preserving bits), gathers the survivors of the row's
// bound from the chunk slots, ranks them in shared memory with branch-free comparisons,
// and draws in fp32 across its lanes (a prefix sum of the k probabilities, then ballots for
// the top-p cut and the inverse CDF): no CTA barrier on the way.  A row whose chunk slots
// overflowed, or with more survivors than a warp holds, is flagged and its exact top-k
// taken afterwards by the whole CTA (a radix select over its logits).
#include "ls_device.cuh"
#include "ls_draw.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr int kSampThreads = 256;
constexpr int kSampWarps = kSampThreads / 32;  // rows per CTA
constexpr int kSampWarpCap = 128;              // survivors a warp holds for its row
constexpr int kSampRounds = 4;                  // gathers of a row's survivors, each with a higher bound
constexpr int kSampHdr = 128;                  // chunk headers a warp keeps in shared memory

struct __align__(16) SampSmem {
  unsigned int gmax[kSampWarps][64];  // group maxima as order-preserving bits
  float cm[kSampWarps][kSampHdr];     // chunk max and survivor count of the first chunks
  int cn[kSampWarps][kSampHdr];
  float cx[kSampWarps][kSampWarpCap];  // survivors (x, token)
  int cv[kSampWarps][kSampWarpCap];
  float tx[kSampWarps][kMaxK];  // the top-k, best first
  int tv[kSampWarps][kMaxK];
  int n[kSampWarps];
  int path[kSampWarps];
  float lse[kSampWarps];
  float R[kSampWarps];
  // exact path (whole CTA, one row at a time)
  float ex[kMaxK];
  int ev[kMaxK];
  int xn;
  unsigned int hist[256];
  unsigned int prefix, pmask;
  int need;
  int wc[kSampWarps];
};

__device__ __forceinline__ void merge_ms(float& M, float& S, float mo, float so) {
  const float Mn = fmaxf(M, mo);
  if (Mn != -INFINITY)
    S = (M == -INFINITY ? 0.0f : S * exp2f((M - Mn) * kLog2e)) + (mo == -INFINITY ? 0.0f : so * exp2f((mo - Mn) * kLog2e));
  M = Mn;
}

// a ranks before b: larger value first, then smaller token
__device__ __forceinline__ bool before(float xa, int va, float xb, int vb) {
  return (xa > xb) | ((xa == xb) & (va < vb));
}

// The draw of one row by one warp from its top-k (tx/tv, best first).
__device__ __forceinline__ void draw(const SampleParams& p, const float* tx, const int* tv, float lse, float u,
                                     int r) {
  draw_topk(tx, tv, p.k, p.top_p, lse, u, r, p.out_token, p.out_logprob);
}

// Exact top-k of row r without the candidate slots, by the whole CTA: radix select of the
// k-th largest value (8 bits at a time from the top), then every element above it and the
// first equal ones in token order.  Leaves exactly k candidates in sm.ex / sm.ev.
template <int DT, bool BIAS>
__device__ void exact_candidates(const SampleParams& p, SampSmem& sm, int r) {
  constexpr int ES = Traits<DT>::kBytes;
  const int K = p.k, V = p.vocab, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned char* rowp = static_cast<const unsigned char*>(p.logits) + (size_t)r * V * ES;
  auto load_x = [&](int v) -> float {
    float x = load_elem<DT>(rowp + (size_t)v * ES);
    if constexpr (BIAS) x += __ldg(p.bias + v);
    return x;
  };
  if (tid == 0) {
    sm.prefix = 0;
    sm.pmask = 0;
    sm.need = K;
    sm.xn = 0;
  }
  __syncthreads();
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kSampThreads) sm.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = sm.prefix, pmask = sm.pmask;
    for (int v = tid; v < V; v += kSampThreads) {
      const uint32_t o = float_ord(load_x(v));
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
  const int need_eq = sm.need;  // equal elements to take, in token order
  for (int v = tid; v < V; v += kSampThreads) {
    const float x = load_x(v);
    if (float_ord(x) > tkey) {
      const int pos = atomicAdd(&sm.xn, 1);
      if (pos < kMaxK) {
        sm.ex[pos] = x;
        sm.ev[pos] = v;
      }
    }
  }
  __syncthreads();
  int taken = 0;
  for (int base = 0; base < V && taken < need_eq; base += kSampThreads) {
    const int v = base + tid;
    float x = 0.0f;
    bool eq = false;
    if (v < V) {
      x = load_x(v);
      eq = float_ord(x) == tkey;
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) sm.wc[warp] = __popc(ballot);
    __syncthreads();
    int before_w = 0, total = 0;
    for (int w = 0; w < kSampWarps; ++w) {
      before_w += (w < warp) ? sm.wc[w] : 0;
      total += sm.wc[w];
    }
    const int off = taken + before_w + __popc(ballot & ((1u << lane) - 1u));
    if (eq && off < need_eq) {
      const int pos = atomicAdd(&sm.xn, 1);
      if (pos < kMaxK) {
        sm.ex[pos] = x;
        sm.ev[pos] = v;
      }
    }
    taken += total;
    __syncthreads();
  }
}

// A warp's full list of entries (lx, lv): the k-th largest x among its n entries (n >= k),
// the larger of it and R as the new bound, and the entries at or above that bound kept in
// order.  Returns (bound, kept count as int bits).  Out of line: it is called from unrolled
// loops.
__device__ __noinline__ float2 list_tighten(float* lx, int* lv, int n, int K, float R) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  float kth = -INFINITY;
  for (int i = lane; i < n; i += 32) {
    const float xi = lx[i];
    int gt = 0, ge = 0;
    for (int q = 0; q < n; ++q) {
      gt += lx[q] > xi;
      ge += lx[q] >= xi;
    }
    if (gt < K && ge >= K) kth = xi;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kth = fmaxf(kth, __shfl_xor_sync(0xffffffffu, kth, o));
  R = fmaxf(R, kth);
  int out = 0;
  for (int b0 = 0; b0 < n; b0 += 32) {
    const int i = b0 + lane;
    const float xi = i < n ? lx[i] : -INFINITY;
    const int vi = i < n ? lv[i] : 0;
    const bool keep = i < n && xi >= R;
    const unsigned bm = __ballot_sync(0xffffffffu, keep);
    __syncwarp();
    if (keep) {
      lx[out + __popc(bm & lt_mask)] = xi;
      lv[out + __popc(bm & lt_mask)] = vi;
    }
    out += __popc(bm);
    __syncwarp();
  }
  return make_float2(R, __int_as_float(out));
}

// Exact top-k of row r by warp w alone: one pass over the row in 16-byte vectors keeps the
// entries x >= R (the row's R-top-k, never above its k-th largest) in the warp's list; a full
// list raises R to the k-th largest of its entries (elements of the row, so still a lower bound)
// and keeps those at or above it.  The list's top-k (larger x, then smaller token) go to
// sm.tx / sm.tv[w].  Returns false when ties at the bound overflow the list.
template <int DT, bool BIAS>
__device__ bool exact_row_warp(const SampleParams& p, SampSmem& sm, int w, int r) {
  constexpr int ES = Traits<DT>::kBytes;
  constexpr int VEC = Traits<DT>::kVec;
  const int K = p.k, V = p.vocab, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  float* lx = sm.cx[w];
  int* lv = sm.cv[w];
  float R = sm.R[w];
  int n = 0;
  bool full = false;
  auto tighten = [&]() {
    const float2 rn = list_tighten(lx, lv, n, K, R);
    R = rn.x;
    n = __float_as_int(rn.y);
  };
  auto append = [&](bool take, float x, int v) {
    unsigned m = __ballot_sync(0xffffffffu, take);
    if (n + __popc(m) > kSampWarpCap) {
      tighten();
      m = __ballot_sync(0xffffffffu, take && x >= R);
      if (n + __popc(m) > kSampWarpCap) {
        full = true;
        return;
      }
    }
    if ((m >> lane) & 1u) {
      lx[n + __popc(m & lt_mask)] = x;
      lv[n + __popc(m & lt_mask)] = v;
    }
    n += __popc(m);
  };
  const unsigned char* rowp = static_cast<const unsigned char*>(p.logits) + (size_t)r * V * ES;
  const int lead = (int)(reinterpret_cast<uintptr_t>(rowp) & 15);
  const uint4* rb = reinterpret_cast<const uint4*>(rowp - lead);
  const int row_bytes = V * ES;
  const int nv = (lead + row_bytes + 15) >> 4;
  // 16-byte vectors covering the row (the first may start before it, the last end after it),
  // four per lane in flight
  for (int v0 = 0; v0 < nv && !full; v0 += 128) {
    uint4 d[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int jv = v0 + 32 * q + lane;
      d[q] = jv < nv ? __ldcs(rb + jv) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const int jv = v0 + 32 * q + lane;
      float xs[VEC];
      const uint4 dv = q == 0 ? d[0] : (q == 1 ? d[1] : (q == 2 ? d[2] : d[3]));  // no local array
      unpack<DT>(dv, xs);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const int byte = jv * 16 + e * ES - lead;
        const bool in = jv < nv && byte >= 0 && byte < row_bytes;
        const int v = byte / ES;
        float x = xs[e];
        if constexpr (BIAS) x += in ? __ldg(p.bias + v) : 0.0f;
        append(in && x >= R, x, v);
      }
    }
  }
  if (full || n < K) return false;
  __syncwarp();
  for (int i = lane; i < n; i += 32) {
    const float xi = lx[i];
    const int vi = lv[i];
    int rank = 0;
    for (int q = 0; q < n; ++q) rank += before(lx[q], lv[q], xi, vi);
    if (rank < K) {
      sm.tx[w][rank] = xi;
      sm.tv[w][rank] = vi;
    }
  }
  return true;
}

template <int DT, bool BIAS>
__global__ void __launch_bounds__(kSampThreads, 1) sample_select_kernel(const SampleParams p) {
  __shared__ SampSmem sm;
  const int K = p.k, nc = p.nc, G = p.groups, C = p.slot_cap;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int r = blockIdx.x * kSampWarps + w;
  const bool row_ok = r < p.rows;
  const float u = row_ok ? p.u[r] : 0.0f;  // not written by K1: read before waiting on it
  sm.gmax[w][lane] = float_ord(-INFINITY);
  sm.gmax[w][lane + 32] = float_ord(-INFINITY);
  if (lane == 0) {
    sm.n[w] = 0;
    sm.path[w] = 0;
  }
  grid_dependency_wait();  // K1's records and slots are complete and visible
  __syncwarp();
  int path = 0;
  if (row_ok) {
    const long long u0 = (long long)r * nc;
    auto rec = [&](int c) { return reinterpret_cast<const float*>(p.rec + (size_t)(u0 + c) * p.rec_stride); };
    // 1. (max, sum of exp) and the group maxima over the row's chunks
    float m = -INFINITY, s = 0.0f;
    bool ovf = false;
    // G <= 8: the group maxima in registers (two vector loads per chunk, then a shuffle
    // tree); more groups go through shared-memory atomics
    float g8[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) g8[g] = -INFINITY;
    for (int c = lane; c < nc; c += 32) {
      const float4* r4 = reinterpret_cast<const float4*>(rec(c));
      const float4 h = __ldcg(r4);
      const int cnt = __float_as_int(h.x);
      ovf |= cnt > C;
      merge_ms(m, s, h.y, h.z);
      if (c < kSampHdr) {
        sm.cm[w][c] = h.y;
        sm.cn[w][c] = cnt;
      }
      if (G <= 8) {
        const float4 ga = __ldcg(r4 + 1);
        const float4 gb = G > 4 ? __ldcg(r4 + 2) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        g8[0] = fmaxf(g8[0], ga.x);
        g8[1] = fmaxf(g8[1], ga.y);
        g8[2] = fmaxf(g8[2], ga.z);
        g8[3] = fmaxf(g8[3], ga.w);
        g8[4] = fmaxf(g8[4], gb.x);
        g8[5] = fmaxf(g8[5], gb.y);
        g8[6] = fmaxf(g8[6], gb.z);
        g8[7] = fmaxf(g8[7], gb.w);
      } else {
        for (int g = 0; g < G; ++g) atomicMax(&sm.gmax[w][g], float_ord(__ldcg(rec(c) + 4 + g)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, m, o);
      const float so = __shfl_xor_sync(0xffffffffu, s, o);
      merge_ms(m, s, mo, so);
    }
    ovf = __any_sync(0xffffffffu, ovf);
    float a, b, gmin = INFINITY;
    if (G <= 8) {
#pragma unroll 1
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int g = 0; g < 8; ++g) g8[g] = fmaxf(g8[g], __shfl_xor_sync(0xffffffffu, g8[g], o));
      }
#pragma unroll
      for (int g = 0; g < 8; ++g) gmin = g < G ? fminf(gmin, g8[g]) : gmin;
      float v = g8[0];
#pragma unroll
      for (int g = 1; g < 8; ++g) v = lane == g ? g8[g] : v;
      a = lane < G ? v : -INFINITY;
      b = -INFINITY;
    } else {
      __syncwarp();
      a = lane < G ? ord_float(sm.gmax[w][lane]) : -INFINITY;
      b = lane + 32 < G ? ord_float(sm.gmax[w][lane + 32]) : -INFINITY;
    }
    // R-top-k: the k-th largest of the G group maxima (ties by group index); with k group
    // maxima in registers it is the least of them
    float R = gmin;
    if (!(G <= 8 && G == K)) {
      int ra = 0, rb = 0;
#pragma unroll 1
      for (int q = 0; q < min(G, 32); ++q) {
        const float wa = __shfl_sync(0xffffffffu, a, q);
        const float wb = __shfl_sync(0xffffffffu, b, q);
        const bool qb = q + 32 < G;  // only the G real groups are ranked
        ra += ((wa > a) | ((wa == a) & (q < lane))) + (qb & (wb > a));
        rb += (wa >= b) + (qb & ((wb > b) | ((wb == b) & (q < lane))));
      }
      const unsigned hit = __ballot_sync(0xffffffffu, ((lane < G) & (ra == K - 1)) | ((lane + 32 < G) & (rb == K - 1)));
      const int hl = __ffs(hit) - 1;
      const float va = __shfl_sync(0xffffffffu, a, hl & 31), vb = __shfl_sync(0xffffffffu, b, hl & 31);
      const int rah = __shfl_sync(0xffffffffu, ra, hl & 31);
      R = rah == K - 1 ? va : vb;
    }
    const float lse = m == -INFINITY ? -INFINITY : m + logf(s);
    path = ovf ? 1 : 0;
    if (p.flags & kFlagForceExact) path = 2;
    // 2. survivors of the row's bound from the chunks whose max reaches it.  When they
    // outnumber the warp's list, the k-th largest of the entries it holds (elements of the
    // row, so still a lower bound of its k-th largest) becomes the bound and the gather runs
    // again, a few times at most.
    for (int round = 0; path == 0 && round < kSampRounds; ++round) {
      if (round > 0) {
        const int held = min(sm.n[w], kSampWarpCap);
        float kth = -INFINITY;
        for (int i = lane; i < held; i += 32) {
          const float xi = sm.cx[w][i];
          int gt = 0, ge = 0;
          for (int q = 0; q < held; ++q) {
            const float xq = sm.cx[w][q];
            gt += xq > xi;
            ge += xq >= xi;
          }
          if (gt < K && ge >= K) kth = xi;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kth = fmaxf(kth, __shfl_xor_sync(0xffffffffu, kth, o));
        R = fmaxf(R, kth);
        __syncwarp();
        if (lane == 0) sm.n[w] = 0;
        __syncwarp();
      }
      for (int c = lane; c < nc; c += 32) {
        float mc;
        int cnt;
        if (c < kSampHdr) {
          mc = sm.cm[w][c];
          cnt = sm.cn[w][c];
        } else {
          const float4 h = __ldcg(reinterpret_cast<const float4*>(rec(c)));
          mc = h.y;
          cnt = __float_as_int(h.x);
        }
        const int n = mc >= R ? min(cnt, C) : 0;
        const CandSlot* sl = p.slots + (size_t)(u0 + c) * C;
        for (int s0 = 0; s0 < n; s0 += 4) {
          int2 raw[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            raw[t] = s0 + t < n ? __ldcg(reinterpret_cast<const int2*>(sl + s0 + t)) : make_int2((int)0xff800000u, 0);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float x = __int_as_float(raw[t].x);
            if ((s0 + t < n) & (x >= R)) {
              const int pos = atomicAdd(&sm.n[w], 1);
              if (pos < kSampWarpCap) {
                sm.cx[w][pos] = x;
                sm.cv[w][pos] = raw[t].y;
              }
            }
          }
        }
      }
      __syncwarp();
      if (sm.n[w] <= kSampWarpCap) break;
    }
    if (path == 0) {
      const int n = sm.n[w];
      if (n > kSampWarpCap || n < K) path = 3;
      if (path == 0) {
        // 3. the exact top-k among the survivors, best first
        for (int i = lane; i < n; i += 32) {
          const float xi = sm.cx[w][i];
          const int vi = sm.cv[w][i];
          int r0 = 0, r1 = 0, q = 0;
#pragma unroll 1
          for (; q + 1 < n; q += 2) {
            r0 += before(sm.cx[w][q], sm.cv[w][q], xi, vi);
            r1 += before(sm.cx[w][q + 1], sm.cv[w][q + 1], xi, vi);
          }
          if (q < n) r0 += before(sm.cx[w][q], sm.cv[w][q], xi, vi);
          if (r0 + r1 < K) {
            sm.tx[w][r0 + r1] = xi;
            sm.tv[w][r0 + r1] = vi;
          }
        }
        __syncwarp();
        // 4. the draw
        draw(p, sm.tx[w], sm.tv[w], lse, u, r);
      }
    }
    if (lane == 0) {
      RowStat st;
      st.lse = lse;
      st.rtopk = R;
      st.ncand = path == 0 ? sm.n[w] : -1;
      st.pad = 0;
      p.rowstat[r] = st;
      p.bstat[r] = path;
      sm.path[w] = path;
      sm.lse[w] = lse;
      sm.R[w] = R;
    }
  }
  // rows that need the exact top-k: first each warp alone over its own row (its entries
  // x >= R in the warp's list, the bound raised to the k-th largest of the list whenever it
  // fills); only a row whose ties at the bound overflow the list takes the whole CTA after.
  __syncwarp();
  if (row_ok && sm.path[w] != 0 && exact_row_warp<DT, BIAS>(p, sm, w, r)) {
    __syncwarp();
    draw(p, sm.tx[w], sm.tv[w], sm.lse[w], u, r);
    __syncwarp();
    if (lane == 0) sm.path[w] = 0;
  }
  __syncthreads();
  for (int w2 = 0; w2 < kSampWarps; ++w2) {
    if (sm.path[w2] == 0) continue;  // CTA-uniform
    const int r2 = blockIdx.x * kSampWarps + w2;
    exact_candidates<DT, BIAS>(p, sm, r2);
    if (w == 0) {
      // rank the k candidates (lanes hold entries lane and lane + 32)
      for (int i = lane; i < K; i += 32) {
        const float xi = sm.ex[i];
        const int vi = sm.ev[i];
        int rk = 0;
        for (int q = 0; q < K; ++q) rk += before(sm.ex[q], sm.ev[q], xi, vi);
        sm.tx[w2][rk] = xi;
        sm.tv[w2][rk] = vi;
      }
      __syncwarp();
      draw(p, sm.tx[w2], sm.tv[w2], sm.lse[w2], p.u[r2], r2);
    }
    __syncthreads();
  }
}

template <int DT, bool BIAS>
cudaError_t launch_t(const SampleParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.rows + kSampWarps - 1) / kSampWarps));
  cfg.blockDim = dim3(kSampThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_select_kernel<DT, BIAS>, p);
}

}  // namespace

cudaError_t launch_sample_select(const SampleParams& p, int dtype, cudaStream_t stream) {
  const bool bias = p.bias != nullptr;
  switch (dtype) {
    case DT_F32: return bias ? launch_t<DT_F32, true>(p, stream) : launch_t<DT_F32, false>(p, stream);
    case DT_F16: return bias ? launch_t<DT_F16, true>(p, stream) : launch_t<DT_F16, false>(p, stream);
    case DT_BF16: return bias ? launch_t<DT_BF16, true>(p, stream) : launch_t<DT_BF16, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsb
