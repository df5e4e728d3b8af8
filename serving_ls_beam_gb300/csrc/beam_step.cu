// Beam-search step kernel: fused first traversal (log_sum_exp + R-top-k) and second
// traversal (threshold filter into the candidate queue) per chunk of a beam's logits,
// with the per-batch fine rank run by whichever CTA finishes that batch's last chunk.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), hierarchical decoding
// section — first traversal (k groups, min of the group maxima = R-top-k <= true k-th
// largest; log_sum_exp in the same pass), second traversal (keep logits >= R-top-k,
// rescore as beam_score + logit - lse, queue them), then one sort of the short queue
// per batch for the exact top-k.
//
// GB300 design (differs from the article's two full traversals of each row):
//  * A row is cut into `nc` chunks.  A persistent CTA streams its chunks through a
//    two-stage shared-memory ring filled by 1-D bulk (TMA) copies, so the logits are
//    read from HBM exactly once and the "second traversal" re-reads registers.
//  * R-top-k is taken per chunk: the chunk's k-th largest group max bounds from below
//    every element of the row's top-k that lies in the chunk (such an element is also
//    in the chunk's own top-k).  The fine rank then re-applies the row-level R-top-k
//    (group maxima merged over chunks), so the surviving candidate set is exactly the
//    article's.  Each chunk writes its candidates to its own fixed slots (no global
//    atomics on a shared queue); the batch id is the slot region, not a float offset.
//  * No second kernel: the CTA whose arrival completes a batch's chunk count ranks
//    that batch's candidates in shared memory while its next chunks keep loading.
//  * If a chunk overflows its slots, the batch's fine rank falls back to an exact
//    radix select over the batch's logits, so the result never depends on capacity.
#include <cuda/atomic>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

constexpr int kStages = 2;
constexpr long long kDrainLimitNs = 2000000000LL;  // 2 s for copies already in flight

enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };
enum { ROW_LIVE = 0, ROW_FIN = 1, ROW_DEAD = 2 };

template <int DT>
struct Traits;
template <>
struct Traits<DT_F32> {
  static constexpr int kVec = 4, kBytes = 4;
  static constexpr uint32_t kNegInfWord = 0xff800000u;
};
template <>
struct Traits<DT_F16> {
  static constexpr int kVec = 8, kBytes = 2;
  static constexpr uint32_t kNegInfWord = 0xfc00fc00u;
};
template <>
struct Traits<DT_BF16> {
  static constexpr int kVec = 8, kBytes = 2;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;
};

template <int DT>
__device__ __forceinline__ void unpack(const uint4& d, float (&x)[Traits<DT>::kVec]) {
  if constexpr (DT == DT_F32) {
    x[0] = __uint_as_float(d.x);
    x[1] = __uint_as_float(d.y);
    x[2] = __uint_as_float(d.z);
    x[3] = __uint_as_float(d.w);
  } else {
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f;
      if constexpr (DT == DT_F16) {
        __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
        f = __half22float2(h);
      } else {
        __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
        f = __bfloat1622float2(h);
      }
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

template <int DT>
__device__ __forceinline__ float load_elem(const unsigned char* p) {
  if constexpr (DT == DT_F32) {
    return __ldg(reinterpret_cast<const float*>(p));
  } else if constexpr (DT == DT_F16) {
    return __half2float(__ldg(reinterpret_cast<const __half*>(p)));
  } else {
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p)));
  }
}

struct RowSel {
  double c;  // beam_score - lse
  float rtopk;
  float lse;
  int kind;
  int ncand;
};

struct __align__(16) Smem {
  unsigned long long bar[kStages];
  float wm[kWarps];
  float wsum[kWarps];
  float wgm[kWarps][32];
  float gmax[64];
  float rthr;
  int cnt;
  int last;
  int abort;
  int refilter;
  float thrmax[kThreads];
  // fine rank
  int nsel, big, ovf, nbest, nrl;
  int wc[kWarps];
  unsigned int hist[256];
  unsigned int prefix, pmask;
  int need;
  RowSel row[kMaxK];
  float selg[kWarps][64];
  Key sel[kSelCap];
  Key mg[2 * kMaxK];
  Key best[kMaxK];
  Key rl[kMaxK];
};

constexpr size_t smem_ctl_bytes() { return (sizeof(Smem) + 127) / 128 * 128; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// k-th largest (1-based) of vals[0..n), n <= 64, computed by one warp; all lanes return it.
__device__ __forceinline__ float warp_kth_largest(const float* vals, int n, int k) {
  const int lane = threadIdx.x & 31;
  float res = -INFINITY;
  for (int g = lane; g < n; g += 32) {
    const float v = vals[g];
    int rank = 0;
    for (int q = 0; q < n; ++q) {
      const float w = vals[q];
      rank += (w > v) || (w == v && q < g);
    }
    if (rank == k - 1) res = v;
  }
  // exactly one lane holds the value; the others hold -inf
  return warp_max(res);
}

__device__ __forceinline__ const float* rec_ptr(const StepParams& p, long long u) {
  return reinterpret_cast<const float*>(p.rec + (size_t)u * p.rec_stride);
}

__device__ __forceinline__ void write_output(const StepParams& p, int b, int r, const Key& key) {
  const int o = b * p.k + r;
  const int parent = key_parent(key);
  const int token = key_token(key);
  p.out_token[o] = token;
  p.out_parent[o] = parent;
  p.out_score[o] = key_score(key);
  if (p.out_finished) {
    const bool fin = p.finished && p.finished[b * p.k + parent];
    p.out_finished[o] = (fin || token == p.eos) ? 1 : 0;
  }
}

// Sort mg[0..n) ascending by key (n a power of two <= 2*kMaxK); all threads call it.
__device__ void bitonic_sort(Key* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int q = i ^ stride;
        if (q > i) {
          const bool up = (i & size) == 0;
          const Key x = a[i], y = a[q];
          if (key_less(y, x) == up) {
            a[i] = y;
            a[q] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Merge sm.rl[0..nrl) into sm.best[0..nbest), keeping the K smallest keys.
__device__ void merge_into_best(Smem& sm, int K) {
  const int nb = sm.nbest, nr = sm.nrl;
  const int tot = nb + nr;
  int n = 1;
  while (n < tot) n <<= 1;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    Key k;
    if (i < nb) {
      k = sm.best[i];
    } else if (i < tot) {
      k = sm.rl[i - nb];
    } else {
      k.hi = ~0ull;
      k.lo = ~0ull;
    }
    sm.mg[i] = k;
  }
  __syncthreads();
  bitonic_sort(sm.mg, n);
  const int keep = tot < K ? tot : K;
  for (int i = threadIdx.x; i < keep; i += kThreads) sm.best[i] = sm.mg[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    sm.nbest = keep;
    sm.nrl = 0;
  }
  __syncthreads();
}

// Exact fine rank of batch b without the candidate queue: per live row, a radix select
// of its top-K logits (order: larger x first, then smaller token id), merged across rows.
template <int DT, bool BIAS>
__device__ void exact_select(const StepParams& p, Smem& sm, int b, int path) {
  constexpr int ES = Traits<DT>::kBytes;
  const int K = p.k, V = p.vocab;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sm.nbest = 0;
    sm.nrl = 0;
  }
  __syncthreads();
  for (int j = 0; j < K; ++j) {
    const RowSel rs = sm.row[j];
    const int row = b * K + j;
    if (rs.kind == ROW_FIN) {
      if (tid == 0) {
        sm.rl[0] = make_key(p.beam[row], j, 0.0f, p.eos);
        sm.nrl = 1;
      }
      __syncthreads();
      merge_into_best(sm, K);
      continue;
    }
    if (rs.kind == ROW_DEAD) {
      for (int v = tid; v < K; v += kThreads) sm.rl[v] = make_key(-INFINITY, j, 0.0f, v);
      if (tid == 0) sm.nrl = K;
      __syncthreads();
      merge_into_best(sm, K);
      continue;
    }
    const unsigned char* rowp = static_cast<const unsigned char*>(p.logits) + (size_t)row * V * ES;
    auto load_x = [&](int v) -> float {
      float x = load_elem<DT>(rowp + (size_t)v * ES);
      if constexpr (BIAS) x += __ldg(p.bias + v);
      return x;
    };
    // radix select of the K-th largest order key, 8 bits at a time from the top
    if (tid == 0) {
      sm.prefix = 0;
      sm.pmask = 0;
      sm.need = K;
    }
    __syncthreads();
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kThreads) sm.hist[i] = 0;
      __syncthreads();
      const uint32_t prefix = sm.prefix, pmask = sm.pmask;
      for (int v = tid; v < V; v += kThreads) {
        const uint32_t o = float_ord(load_x(v));
        if ((o & pmask) == prefix) atomicAdd(&sm.hist[(o >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        int need = sm.need;
        unsigned int cum = 0;
        int d = 255;
        for (; d > 0; --d) {
          if (cum + sm.hist[d] >= (unsigned)need) break;
          cum += sm.hist[d];
        }
        sm.need = need - (int)cum;
        sm.prefix = prefix | ((uint32_t)d << shift);
        sm.pmask = pmask | (255u << shift);
      }
      __syncthreads();
    }
    const uint32_t tkey = sm.prefix;
    const int need_eq = sm.need;  // ties at the threshold to take, in token order
    // strictly greater: fewer than K of them, order irrelevant
    for (int v = tid; v < V; v += kThreads) {
      const float x = load_x(v);
      if (float_ord(x) > tkey) {
        const int pos = atomicAdd(&sm.nrl, 1);
        if (pos < kMaxK) sm.rl[pos] = make_key((float)(rs.c + (double)x), j, x, v);
      }
    }
    __syncthreads();
    // ties: the first need_eq of them by token id
    int taken = 0;
    for (int base = 0; base < V && taken < need_eq; base += kThreads) {
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
      int before = 0, total = 0;
      for (int w = 0; w < kWarps; ++w) {
        before += (w < warp) ? sm.wc[w] : 0;
        total += sm.wc[w];
      }
      const int off = taken + before + __popc(ballot & ((1u << lane) - 1u));
      if (eq && off < need_eq) {
        const int pos = atomicAdd(&sm.nrl, 1);
        if (pos < kMaxK) sm.rl[pos] = make_key((float)(rs.c + (double)x), j, x, v);
      }
      taken += total;
      __syncthreads();
    }
    if (tid == 0 && sm.nrl > kMaxK) sm.nrl = kMaxK;  // cannot happen: greater + ties == K
    __syncthreads();
    merge_into_best(sm, K);
  }
  for (int r = tid; r < K && r < sm.nbest; r += kThreads) write_output(p, b, r, sm.best[r]);
  for (int j = tid; j < K; j += kThreads) {
    const RowSel rs = sm.row[j];
    RowStat st;
    st.lse = rs.kind == ROW_FIN ? __int_as_float(0x7fc00000) : rs.lse;
    st.rtopk = rs.rtopk;
    st.ncand = -1;
    st.pad = 0;
    p.rowstat[b * K + j] = st;
  }
  if (tid == 0) p.bstat[b] = path;
}

// Fine rank of batch b, run by the CTA that completed the batch.  All threads call it.
template <int DT, bool BIAS>
__device__ __noinline__ void select_batch(const StepParams& p, Smem& sm, int b) {
  const int K = p.k, nc = p.nc, G = p.groups, C = p.slot_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sm.nsel = 0;
    sm.big = 0;
    sm.ovf = 0;
  }
  __syncthreads();
  // 1. per-row lse, R-top-k and score offset from the chunk records
  for (int j = warp; j < K; j += kWarps) {
    const int row = b * K + j;
    const bool fin = p.finished && p.finished[row];
    const float beam = p.beam[row];
    if (fin) {
      if (lane == 0) {
        RowSel rs;
        rs.c = 0.0;
        rs.rtopk = __int_as_float(0x7fc00000);
        rs.lse = __int_as_float(0x7fc00000);
        rs.kind = ROW_FIN;
        rs.ncand = 1;
        sm.row[j] = rs;
      }
      continue;
    }
    const long long u0 = (long long)row * nc;
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(rec_ptr(p, u0 + c) + 1));
    M = warp_max(M);
    double S = 0.0;
    bool ovf = false;
    for (int c = lane; c < nc; c += 32) {
      const float* r = rec_ptr(p, u0 + c);
      const float mc = __ldcg(r + 1);
      const float sc = __ldcg(r + 2);
      const int cnt = __ldcg(reinterpret_cast<const int*>(r));
      if (mc != -INFINITY) S += (double)sc * exp((double)mc - (double)M);
      ovf |= cnt > C;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    ovf = __any_sync(0xffffffffu, ovf);
    for (int g = lane; g < G; g += 32) {
      float gm = -INFINITY;
      for (int c = 0; c < nc; ++c) gm = fmaxf(gm, __ldcg(rec_ptr(p, u0 + c) + 4 + g));
      sm.selg[warp][g] = gm;
    }
    __syncwarp();
    const float rt = warp_kth_largest(sm.selg[warp], G, K);
    if (lane == 0) {
      const double lse = (M == -INFINITY) ? -(double)INFINITY : (double)M + log(S);
      RowSel rs;
      rs.lse = (float)lse;
      rs.rtopk = rt;
      rs.ncand = 0;
      if (M == -INFINITY || beam == -INFINITY) {
        rs.kind = ROW_DEAD;
        rs.c = -(double)INFINITY;
      } else {
        rs.kind = ROW_LIVE;
        rs.c = (double)beam - lse;
      }
      sm.row[j] = rs;
      if (ovf) sm.ovf = 1;
    }
    __syncwarp();
  }
  __syncthreads();
  int path = 0;
  if (sm.ovf) path = 1;
  if (p.flags & kFlagForceExact) path = 2;
  if (path == 0) {
    // 2. survivors of the row-level R-top-k, rescored: beam_score + x - lse
    for (int pair = warp; pair < K * nc; pair += kWarps) {
      const int j = pair / nc;
      const RowSel& rs = sm.row[j];
      if (rs.kind != ROW_LIVE) continue;
      const long long u = (long long)(b * K + j) * nc + (pair - j * nc);
      const int cnt = min(__ldcg(reinterpret_cast<const int*>(rec_ptr(p, u))), C);
      const float rt = rs.rtopk;
      const double cj = rs.c;
      for (int q = lane; q < cnt; q += 32) {
        const int2 raw = __ldcg(reinterpret_cast<const int2*>(p.slots + (size_t)u * C + q));
        const float x = __int_as_float(raw.x);
        if (x >= rt) {
          const Key key = make_key((float)(cj + (double)x), j, x, raw.y);
          const int pos = atomicAdd(&sm.nsel, 1);
          if (pos < kSelCap)
            sm.sel[pos] = key;
          else
            sm.big = 1;
          atomicAdd(&sm.row[j].ncand, 1);
        }
      }
    }
    for (int idx = tid; idx < K * K; idx += kThreads) {
      const int j = idx / K, v = idx - (idx / K) * K;
      const int kind = sm.row[j].kind;
      if (kind == ROW_FIN && v == 0) {
        const int pos = atomicAdd(&sm.nsel, 1);
        if (pos < kSelCap)
          sm.sel[pos] = make_key(p.beam[b * K + j], j, 0.0f, p.eos);
        else
          sm.big = 1;
      } else if (kind == ROW_DEAD) {
        const int pos = atomicAdd(&sm.nsel, 1);
        if (pos < kSelCap)
          sm.sel[pos] = make_key(-INFINITY, j, 0.0f, v);
        else
          sm.big = 1;
        if (v == 0) sm.row[j].ncand = K;
      }
    }
    __syncthreads();
    if (sm.big) path = 3;
  }
  if (path != 0) {
    exact_select<DT, BIAS>(p, sm, b, path);
    return;
  }
  // 3. rank of every survivor among the survivors; the first K are the output
  const int n = sm.nsel;
  for (int i = tid; i < n; i += kThreads) {
    const Key ki = sm.sel[i];
    int rank = 0;
    for (int q = 0; q < n; ++q) rank += key_less(sm.sel[q], ki);
    if (rank < K) write_output(p, b, rank, ki);
  }
  for (int j = tid; j < K; j += kThreads) {
    const RowSel rs = sm.row[j];
    RowStat st;
    st.lse = rs.kind == ROW_FIN ? __int_as_float(0x7fc00000) : rs.lse;
    st.rtopk = rs.rtopk;
    st.ncand = rs.ncand;
    st.pad = 0;
    p.rowstat[b * K + j] = st;
  }
  if (tid == 0) p.bstat[b] = 0;
}

template <int DT, bool BIAS, int VPT>
__global__ void __launch_bounds__(kThreads, 3) beam_step_kernel(const StepParams p) {
  constexpr int VEC = Traits<DT>::kVec;
  constexpr int ES = Traits<DT>::kBytes;
  constexpr uint32_t kStageBytes = VPT * kThreads * 16;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  unsigned char* stages = smem_raw + smem_ctl_bytes();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.k, V = p.vocab, nc = p.nc, G = p.groups, C = p.slot_cap;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&sm.bar[s]), 1);
    sm.cnt = 0;
    sm.last = 0;
    sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const long long units = p.units;
  const long long first = blockIdx.x, step = gridDim.x;
  const long long n_mine = first < units ? (units - first + step - 1) / step : 0;
  const unsigned char* logits = static_cast<const unsigned char*>(p.logits);

  auto unit_live = [&](long long u) -> bool {
    const int row = (int)(u / nc);
    return !(p.finished && p.finished[row]);
  };
  // chunk geometry: [head scalars][n_vec 16-byte vectors][tail scalars]
  struct Geo {
    const unsigned char* g;
    int e0, n_head, n_vec, n_tail;
  };
  auto geometry = [&](long long u) -> Geo {
    Geo q;
    const int row = (int)(u / nc), c = (int)(u - (long long)row * nc);
    q.e0 = c * p.chunk_len;
    const int e1 = min(q.e0 + p.chunk_len, V);
    const int n_el = max(e1 - q.e0, 0);
    q.g = logits + ((size_t)row * V + q.e0) * ES;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(q.g);
    const uintptr_t aend = a0 + (uintptr_t)n_el * ES;
    const uintptr_t A = (a0 + 15) & ~(uintptr_t)15;
    const uintptr_t B = aend & ~(uintptr_t)15;
    if (n_el == 0 || A >= B) {
      q.n_head = n_el;
      q.n_vec = 0;
      q.n_tail = 0;
    } else {
      q.n_head = (int)((A - a0) / ES);
      q.n_vec = (int)((B - A) / 16);
      q.n_tail = (int)((aend - B) / ES);
    }
    return q;
  };

  // producer state, used by thread 0 only
  long long iss_i = 0, n_iss = 0;
  uint64_t policy = 0;
  if (tid == 0) policy = l2_evict_first_policy();
  auto fill = [&](long long n_cons) {
    while (n_iss - n_cons < kStages && iss_i < n_mine) {
      const long long u = first + iss_i * step;
      if (unit_live(u)) {
        const Geo q = geometry(u);
        const int s = (int)(n_iss % kStages);
        const uint32_t bar = smem_addr(&sm.bar[s]);
        const uint32_t bytes = (uint32_t)q.n_vec * 16u;
        mbar_arrive_expect_tx(bar, bytes);
        if (bytes) bulk_load(smem_addr(stages + (size_t)s * kStageBytes), q.g + (size_t)q.n_head * ES, bytes, bar,
                             policy);
        ++n_iss;
      }
      ++iss_i;
    }
  };
  if (tid == 0) fill(0);

  long long n_cons = 0;
  for (long long i = 0; i < n_mine; ++i) {
    const long long u = first + i * step;
    const int row = (int)(u / nc);
    const int b = row / K;
    if (unit_live(u)) {
      const Geo q = geometry(u);
      const int s = (int)(n_cons % kStages);
      // head / tail elements: one per thread, plain loads
      float xe = -INFINITY;
      int ve = 0;
      bool has_x = false;
      if (tid < q.n_head) {
        ve = tid;
        has_x = true;
      } else if (tid - q.n_head < q.n_tail) {
        ve = q.n_head + q.n_vec * VEC + (tid - q.n_head);
        has_x = true;
      }
      if (has_x) {
        xe = load_elem<DT>(q.g + (size_t)ve * ES);
        if constexpr (BIAS) xe += __ldg(p.bias + q.e0 + ve);
      }
      const bool ok = mbar_wait_bounded(smem_addr(&sm.bar[s]), (uint32_t)((n_cons / kStages) & 1), p.spin_limit_ns);
      if (!ok) sm.abort = 1;
      const uint4* sv = reinterpret_cast<const uint4*>(stages + (size_t)s * kStageBytes);
      uint4 d[VPT];
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        const int iv = tid + r * kThreads;
        if (iv < q.n_vec) {
          d[r] = sv[iv];
        } else {
          const uint32_t w = Traits<DT>::kNegInfWord;
          d[r] = make_uint4(w, w, w, w);
        }
      }
      const int vbase = q.e0 + q.n_head;  // token id of vector 0, element 0
      bool bias_vec = false;
      if constexpr (BIAS) bias_vec = ((reinterpret_cast<uintptr_t>(p.bias + vbase)) & 15) == 0;
      auto values = [&](int r, float (&x)[VEC]) {
        unpack<DT>(d[r], x);
        if constexpr (BIAS) {
          const int iv = tid + r * kThreads;
          if (iv < q.n_vec) {
            const float* bp = p.bias + vbase + iv * VEC;
            if (bias_vec) {
#pragma unroll
              for (int e = 0; e < VEC; e += 4) {
                const float4 bb = __ldg(reinterpret_cast<const float4*>(bp + e));
                x[e] += bb.x;
                x[e + 1] += bb.y;
                x[e + 2] += bb.z;
                x[e + 3] += bb.w;
              }
            } else {
#pragma unroll
              for (int e = 0; e < VEC; ++e) x[e] += __ldg(bp + e);
            }
          }
        }
      };
      // first traversal: thread max (= this thread's group contribution), then sum of exp
      float mt = xe;
#pragma unroll
      for (int r = 0; r < VPT; ++r) {
        float x[VEC];
        values(r, x);
#pragma unroll
        for (int e = 0; e < VEC; ++e) mt = fmaxf(mt, x[e]);
      }
      // exp(x - m) as 2^((x - m) * log2 e): the difference is exact for the terms that
      // dominate the sum (x within a factor 2 of m), so large logits keep full precision
      float st = 0.0f;
      if (mt != -INFINITY) {
#pragma unroll
        for (int r = 0; r < VPT; ++r) {
          float x[VEC];
          values(r, x);
#pragma unroll
          for (int e = 0; e < VEC; ++e) st += fast_exp2((x[e] - mt) * kLog2e);
        }
        if (has_x) st += fast_exp2((xe - mt) * kLog2e);
      }
      // warp: combine (max, sum) and the group maxima (group = thread index mod G)
      float m = mt, ssum = st;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, o);
        const float so = __shfl_xor_sync(0xffffffffu, ssum, o);
        const float M = fmaxf(m, mo);
        ssum = (M == -INFINITY) ? 0.0f
                                : ssum * fast_exp2((m - M) * kLog2e) + so * fast_exp2((mo - M) * kLog2e);
        m = M;
      }
      float gmv = mt;
      for (int o = 16; o >= G; o >>= 1) gmv = fmaxf(gmv, __shfl_xor_sync(0xffffffffu, gmv, o));
      if (lane == 0) {
        sm.wm[warp] = m;
        sm.wsum[warp] = ssum;
      }
      if (lane < G) sm.wgm[warp][lane] = gmv;
      __syncthreads();  // BAR1: the stage is consumed (registers hold it)
      if (sm.abort) break;
      if (tid == 0) fill(n_cons + 1);
      float* rec = reinterpret_cast<float*>(p.rec + (size_t)u * p.rec_stride);
      if (warp == 0) {
        float m2 = lane < kWarps ? sm.wm[lane] : -INFINITY;
        float s2 = lane < kWarps ? sm.wsum[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float mo = __shfl_xor_sync(0xffffffffu, m2, o);
          const float so = __shfl_xor_sync(0xffffffffu, s2, o);
          const float M = fmaxf(m2, mo);
          s2 = (M == -INFINITY) ? 0.0f : s2 * fast_exp2((m2 - M) * kLog2e) + so * fast_exp2((mo - M) * kLog2e);
          m2 = M;
        }
        for (int g = lane; g < G; g += 32) {
          float gm = -INFINITY;
          if (G <= 32) {
            for (int w = 0; w < kWarps; ++w) gm = fmaxf(gm, sm.wgm[w][g]);
          } else {
            for (int w = (g >> 5); w < kWarps; w += 2) gm = fmaxf(gm, sm.wgm[w][g & 31]);
          }
          sm.gmax[g] = gm;
          rec[4 + g] = gm;
        }
        __syncwarp();
        const float rt = warp_kth_largest(sm.gmax, G, K);
        if (lane == 0) {
          sm.rthr = rt;
          rec[1] = m2;
          rec[2] = s2;
        }
      }
      __syncthreads();  // BAR2: chunk threshold known
      // second traversal: keep x >= threshold (only threads whose max reaches it can hold one)
      CandSlot* slots = p.slots + (size_t)u * C;
      auto filter = [&](float thr) {
        bool wrote = false;
        if (mt >= thr) {
#pragma unroll
          for (int r = 0; r < VPT; ++r) {
            const int iv = tid + r * kThreads;
            if (iv < q.n_vec) {
              float x[VEC];
              values(r, x);
#pragma unroll
              for (int e = 0; e < VEC; ++e) {
                if (x[e] >= thr) {
                  const int pos = atomicAdd(&sm.cnt, 1);
                  if (pos < C) {
                    CandSlot cs;
                    cs.x = x[e];
                    cs.v = vbase + iv * VEC + e;
                    slots[pos] = cs;
                    wrote = true;
                  }
                }
              }
            }
          }
          if (has_x && xe >= thr) {
            const int pos = atomicAdd(&sm.cnt, 1);
            if (pos < C) {
              CandSlot cs;
              cs.x = xe;
              cs.v = q.e0 + ve;
              slots[pos] = cs;
              wrote = true;
            }
          }
        }
        if (wrote) __threadfence();
      };
      auto publish = [&]() {  // thread 0: chunk count, then arrival on the batch counter
        reinterpret_cast<int*>(rec)[0] = sm.cnt;
        sm.cnt = 0;
        __threadfence();
        cuda::atomic_ref<unsigned int, cuda::thread_scope_device> done(p.done[b]);
        const unsigned int old = done.fetch_add(1u, cuda::std::memory_order_acq_rel);
        sm.last = (old == (unsigned int)(K * nc - 1)) ? 1 : 0;
      };
      filter(sm.rthr);
      __syncthreads();  // BAR3: all candidates of the chunk written
      if (tid == 0) {
        sm.refilter = sm.cnt > C;
        if (!sm.refilter) publish();
      }
      __syncthreads();  // BAR4: last-arrival (or refilter) flag visible
      if (sm.refilter) {
        // Too many survivors for the chunk's slots (heavy tails or ties with k groups):
        // tighten to the k-th largest of the per-thread maxima (kThreads disjoint groups,
        // still a lower bound on the chunk's k-th largest) and filter again.
        sm.thrmax[tid] = mt;
        if (tid == 0) sm.cnt = 0;
        __syncthreads();
        if (warp == 0) {
          float res = -INFINITY;
          for (int g = lane; g < kThreads; g += 32) {
            const float v = sm.thrmax[g];
            int rank = 0;
            for (int q2 = 0; q2 < kThreads; ++q2) {
              const float w2 = sm.thrmax[q2];
              rank += (w2 > v) || (w2 == v && q2 < g);
            }
            if (rank == K - 1) res = v;
          }
          res = warp_max(res);
          if (lane == 0) sm.rthr = res;
        }
        __syncthreads();
        filter(sm.rthr);
        __syncthreads();
        if (tid == 0) publish();
        __syncthreads();  // last-arrival flag visible
      }
      ++n_cons;
    } else {
      if (tid == 0) {
        cuda::atomic_ref<unsigned int, cuda::thread_scope_device> done(p.done[b]);
        const unsigned int old = done.fetch_add(1u, cuda::std::memory_order_acq_rel);
        sm.last = (old == (unsigned int)(K * nc - 1)) ? 1 : 0;
      }
      __syncthreads();  // last-arrival flag visible
    }
    if (sm.last) {
      __threadfence();
      select_batch<DT, BIAS>(p, sm, b);
      __syncthreads();
      if (tid == 0) {
        sm.last = 0;
        p.done[b] = 0u;
      }
      __syncthreads();
    }
  }

  if (sm.abort) {
    // a wait ran out: record it, then let every copy already issued land before exit
    if (tid == 0) {
      atomicOr(p.status, kDevTimeout);
      for (long long n = n_cons; n < n_iss; ++n)
        mbar_wait_bounded(smem_addr(&sm.bar[n % kStages]), (uint32_t)((n / kStages) & 1), kDrainLimitNs);
    }
    __syncthreads();
  }
}

template <int DT, bool BIAS, int VPT>
cudaError_t launch_t(const StepParams& p, int grid, size_t smem, cudaStream_t stream) {
  beam_step_kernel<DT, BIAS, VPT><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int DT, bool BIAS, int VPT>
cudaError_t config_t(size_t smem, int* occ) {
  auto fn = beam_step_kernel<DT, BIAS, VPT>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kThreads, smem);
}

template <int DT, bool BIAS>
cudaError_t dispatch_vpt(bool launch, const StepParams* p, int vpt, int grid, size_t smem, cudaStream_t stream,
                         int* occ) {
  switch (vpt) {
    case 4:
      return launch ? launch_t<DT, BIAS, 4>(*p, grid, smem, stream) : config_t<DT, BIAS, 4>(smem, occ);
    case 6:
      return launch ? launch_t<DT, BIAS, 6>(*p, grid, smem, stream) : config_t<DT, BIAS, 6>(smem, occ);
    case 8:
      return launch ? launch_t<DT, BIAS, 8>(*p, grid, smem, stream) : config_t<DT, BIAS, 8>(smem, occ);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch(bool launch, const StepParams* p, int dtype, bool bias, int vpt, int grid, size_t smem,
                     cudaStream_t stream, int* occ) {
  switch (dtype) {
    case DT_F32:
      return bias ? dispatch_vpt<DT_F32, true>(launch, p, vpt, grid, smem, stream, occ)
                  : dispatch_vpt<DT_F32, false>(launch, p, vpt, grid, smem, stream, occ);
    case DT_F16:
      return bias ? dispatch_vpt<DT_F16, true>(launch, p, vpt, grid, smem, stream, occ)
                  : dispatch_vpt<DT_F16, false>(launch, p, vpt, grid, smem, stream, occ);
    case DT_BF16:
      return bias ? dispatch_vpt<DT_BF16, true>(launch, p, vpt, grid, smem, stream, occ)
                  : dispatch_vpt<DT_BF16, false>(launch, p, vpt, grid, smem, stream, occ);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t beam_step_smem_bytes(int vpt) { return smem_ctl_bytes() + (size_t)kStages * vpt * kThreads * 16; }

cudaError_t beam_step_config(int dtype, bool bias, int vpt, size_t smem, int* occupancy) {
  return dispatch(false, nullptr, dtype, bias, vpt, 0, smem, nullptr, occupancy);
}

cudaError_t launch_beam_step(const StepParams& p, int dtype, int vpt, int grid, size_t smem, cudaStream_t stream) {
  return dispatch(true, &p, dtype, p.bias != nullptr, vpt, grid, smem, stream, nullptr);
}

}  // namespace lsb
