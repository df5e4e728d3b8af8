// Sampling kernel K5: the draw of one token per sequence from the top-k (optionally
// top-p) candidates of its logits, after K1 has streamed every row once.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), decoding section: besides
// beam search, decoding by sampling.  The hierarchical first traversal applies unchanged:
// K1 gives per chunk (max, sum of exp, group maxima) and the chunk's survivors above its
// R-top-k bound; this kernel merges them into the row's log_sum_exp and R-top-k, keeps the
// survivors above that bound, takes the exact top-k among them, and draws by inverse CDF
// at the caller's uniform u.
//
// GB300 design: one CTA per row, launched with programmatic dependent launch behind K1.
// The row's records are merged by all threads (group maxima through shared-memory atomics
// on order-preserving bits), the candidates are ranked in shared memory with branch-free
// comparisons, and the final draw (k <= 64 terms in double) is one thread's loop.  A row
// whose chunk slots overflowed, or with more candidates than fit, takes an exact radix
// select of its top-k over the logits instead.
#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr int kSampThreads = 256;
constexpr int kSampWarps = kSampThreads / 32;
constexpr int kSampCap = 1024;  // candidates held in shared memory

struct __align__(16) SampSmem {
  unsigned int gmax[64];  // group maxima as order-preserving bits
  float wm[kSampWarps], ws[kSampWarps];
  float M, S, R, lse;
  int ovf, n;
  float cx[kSampCap];  // candidates (x, token)
  int cv[kSampCap];
  float tx[kMaxK];  // the top-k, best first
  int tv[kMaxK];
  unsigned int hist[256];
  unsigned int prefix, pmask;
  int need, nsel;
  int wc[kSampWarps];
};

__device__ __forceinline__ void merge_ms(float& M, float& S, float mo, float so) {
  const float Mn = fmaxf(M, mo);
  if (Mn != -INFINITY)
    S = (M == -INFINITY ? 0.0f : S * exp2f((M - Mn) * kLog2e)) + (mo == -INFINITY ? 0.0f : so * exp2f((mo - Mn) * kLog2e));
  M = Mn;
}

// x ranks before y: larger value first, then smaller token
__device__ __forceinline__ bool before(float xa, int va, float xb, int vb) {
  return (xa > xb) | ((xa == xb) & (va < vb));
}

// Rank the sm.n candidates; rank < k goes to position rank of the top-k.
__device__ void rank_candidates(SampSmem& sm, int K) {
  const int n = sm.n;
  for (int i = threadIdx.x; i < n; i += kSampThreads) {
    const float xi = sm.cx[i];
    const int vi = sm.cv[i];
    int r0 = 0, r1 = 0, q = 0;
#pragma unroll 1
    for (; q + 1 < n; q += 2) {
      r0 += before(sm.cx[q], sm.cv[q], xi, vi);
      r1 += before(sm.cx[q + 1], sm.cv[q + 1], xi, vi);
    }
    if (q < n) r0 += before(sm.cx[q], sm.cv[q], xi, vi);
    const int r = r0 + r1;
    if (r < K) {
      sm.tx[r] = xi;
      sm.tv[r] = vi;
    }
  }
}

// Exact top-k of the row without the candidate slots: radix select of the k-th largest
// value (8 bits at a time from the top), then every element above it and the first
// equal ones in token order.  Leaves exactly k candidates in sm.cx / sm.cv.
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
    sm.n = 0;
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
      const int pos = atomicAdd(&sm.n, 1);
      if (pos < kSampCap) {
        sm.cx[pos] = x;
        sm.cv[pos] = v;
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
      const int pos = atomicAdd(&sm.n, 1);
      if (pos < kSampCap) {
        sm.cx[pos] = x;
        sm.cv[pos] = v;
      }
    }
    taken += total;
    __syncthreads();
  }
  if (tid == 0 && sm.n > K) sm.n = K;  // greater + equal taken == k
  __syncthreads();
}

template <int DT, bool BIAS>
__global__ void __launch_bounds__(kSampThreads, 1) sample_select_kernel(const SampleParams p) {
  __shared__ SampSmem sm;
  const int K = p.k, nc = p.nc, G = p.groups, C = p.slot_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const float u = p.u[r];  // not written by K1: read before waiting on it
  if (tid < 64) sm.gmax[tid] = float_ord(-INFINITY);
  if (tid == 0) {
    sm.ovf = 0;
    sm.n = 0;
  }
  grid_dependency_wait();  // K1's records and slots are complete and visible
  __syncthreads();
  const long long u0 = (long long)r * nc;
  auto rec = [&](long long uu) { return reinterpret_cast<const float*>(p.rec + (size_t)uu * p.rec_stride); };
  // 1. (max, sum of exp) over the chunks, the group maxima merged over the chunks
  float m = -INFINITY, s = 0.0f;
  bool ovf = false;
  for (int c = tid; c < nc; c += kSampThreads) {
    const float4 h = __ldcg(reinterpret_cast<const float4*>(rec(u0 + c)));
    ovf |= __float_as_int(h.x) > C;
    merge_ms(m, s, h.y, h.z);
  }
  for (int i = tid; i < nc * G; i += kSampThreads) {
    const int c = i / G, g = i - c * G;
    atomicMax(&sm.gmax[g], float_ord(__ldcg(rec(u0 + c) + 4 + g)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    merge_ms(m, s, mo, so);
  }
  ovf = __any_sync(0xffffffffu, ovf);
  if (lane == 0) {
    sm.wm[warp] = m;
    sm.ws[warp] = s;
    if (ovf) sm.ovf = 1;
  }
  __syncthreads();
  if (warp == 0) {
    float M = lane < kSampWarps ? sm.wm[lane] : -INFINITY, S = lane < kSampWarps ? sm.ws[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, M, o);
      const float so = __shfl_xor_sync(0xffffffffu, S, o);
      merge_ms(M, S, mo, so);
    }
    // R-top-k: the k-th largest of the G group maxima (ties by group index)
    const float a = lane < G ? ord_float(sm.gmax[lane]) : -INFINITY;
    const float b = lane + 32 < G ? ord_float(sm.gmax[lane + 32]) : -INFINITY;
    int ra = 0, rb = 0;
#pragma unroll 1
    for (int q = 0; q < 32; ++q) {
      const float wa = __shfl_sync(0xffffffffu, a, q);
      const float wb = __shfl_sync(0xffffffffu, b, q);
      const bool qa = q < G, qb = q + 32 < G;  // only the G real groups are ranked
      ra += (qa & ((wa > a) | ((wa == a) & (q < lane)))) + (qb & (wb > a));
      rb += (qa & (wa >= b)) + (qb & ((wb > b) | ((wb == b) & (q < lane))));
    }
    const unsigned hit = __ballot_sync(0xffffffffu, ((lane < G) & (ra == K - 1)) | ((lane + 32 < G) & (rb == K - 1)));
    const int hl = __ffs(hit) - 1;
    const float va = __shfl_sync(0xffffffffu, a, hl), vb = __shfl_sync(0xffffffffu, b, hl);
    const int rah = __shfl_sync(0xffffffffu, ra, hl);
    if (lane == 0) {
      sm.M = M;
      sm.S = S;
      sm.R = (hl < G && rah == K - 1) ? va : vb;
      sm.lse = M == -INFINITY ? -INFINITY : M + logf(S);
    }
  }
  __syncthreads();
  const float R = sm.R;
  int path = sm.ovf ? 1 : 0;
  if (p.flags & kFlagForceExact) path = 2;
  if (path == 0) {
    // 2. survivors of the row's R-top-k from the chunks that can hold one
    for (int c = tid; c < nc; c += kSampThreads) {
      const float4 h = __ldcg(reinterpret_cast<const float4*>(rec(u0 + c)));
      const int n = h.y >= R ? min(__float_as_int(h.x), C) : 0;
      const CandSlot* sl = p.slots + (size_t)(u0 + c) * C;
      for (int s0 = 0; s0 < n; s0 += 4) {
        int2 raw[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) raw[t] = s0 + t < n ? __ldcg(reinterpret_cast<const int2*>(sl + s0 + t)) : make_int2((int)0xff800000u, 0);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float x = __int_as_float(raw[t].x);
          if ((s0 + t < n) & (x >= R)) {
            const int pos = atomicAdd(&sm.n, 1);
            if (pos < kSampCap) {
              sm.cx[pos] = x;
              sm.cv[pos] = raw[t].y;
            }
          }
        }
      }
    }
    __syncthreads();
    if (sm.n > kSampCap || sm.n < K) path = 3;
  }
  const int ncand = sm.n;
  __syncthreads();
  if (path != 0) exact_candidates<DT, BIAS>(p, sm, r);
  // 3. the exact top-k, best first
  rank_candidates(sm, K);
  __syncthreads();
  // 4. the draw: cumulative probabilities over the top-k (renormalised), the top-p prefix,
  // then the first candidate whose cumulative probability exceeds u
  if (tid == 0) {
    const double x0 = sm.tx[0];
    double tot = 0.0;
    for (int i = 0; i < K; ++i) tot += exp((double)sm.tx[i] - x0);
    int mk = K;
    double totm = tot;
    if (p.top_p < 1.0f) {
      double acc = 0.0;
      for (int i = 0; i < K; ++i) {
        acc += exp((double)sm.tx[i] - x0);
        if (acc >= (double)p.top_p * tot) {
          mk = i + 1;
          totm = acc;
          break;
        }
      }
    }
    const double target = (double)u * totm;
    double acc = 0.0;
    int pick = mk - 1;
    for (int i = 0; i < mk; ++i) {
      acc += exp((double)sm.tx[i] - x0);
      if (acc > target) {
        pick = i;
        break;
      }
    }
    p.out_token[r] = sm.tv[pick];
    if (p.out_logprob) p.out_logprob[r] = sm.tx[pick] - sm.lse;
    RowStat st;
    st.lse = sm.lse;
    st.rtopk = R;
    st.ncand = path == 0 ? ncand : -1;
    st.pad = 0;
    p.rowstat[r] = st;
    p.bstat[r] = path;
  }
}

template <int DT, bool BIAS>
cudaError_t launch_t(const SampleParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.rows);
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
