// Beam-step kernel K2: the fine rank.  One CTA per batch merges the chunk records of
// that batch's beams, re-applies each beam's row-level R-top-k, rescores the surviving
// candidates and ranks them; the k best are the step's output.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), hierarchical decoding
// section: candidates above R-top-k are rescored as beam_score + logit - log_sum_exp
// and one sort of that short queue per batch gives the exact top-k of every sequence.
//
// GB300 design: launched with programmatic dependent launch behind K1, so its launch
// and prologue overlap K1's last wave; `griddepcontrol.wait` orders it after K1's
// writes.  The queue is short (about a dozen survivors per beam for k = 4), so instead
// of a sort each survivor's rank is counted against all the others in shared memory,
// O(n^2 / threads), and the k with rank < k are written.  A batch whose chunk slots
// overflowed, or with more than kSelCap survivors, takes an exact path that needs no
// queue: a per-beam radix select of the top-k logits, merged across beams.
#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

enum { ROW_LIVE = 0, ROW_FIN = 1, ROW_DEAD = 2 };

struct RowSel {
  ScoreBase c;  // beam_score - log_sum_exp
  float rtopk;
  float lse;
  int kind;
  int ncand;
};

constexpr int kPairTile = 1024;  // (beam, chunk) pairs whose slot counts are scanned at once

struct __align__(16) SelSmem {
  unsigned long long sbar;  // completion of the slot staging copy
  int nsel, big, ovf, nbest, nrl, ptotal, ecnt;
  int pc[kPairTile];   // slots to read per pair of the tile, then their exclusive prefix sums
  float pm[kPairTile];  // chunk max of each (beam, chunk) pair (first tile only)
  int pn[kPairTile];    // survivor count of each pair (first tile only)
  float beam[kMaxK];
  int fin[kMaxK];
  int wsum[kSelWarps];
  int wc[kSelWarps];
  unsigned int hist[256];
  unsigned int prefix, pmask;
  int need;
  RowSel row[kMaxK];
  float selg[kSelWarps][64];
  Key sel[kSelCap];
  Key mg[2 * kMaxK];
  Key best[kMaxK];
  Key rl[kMaxK];
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// k-th largest (1-based) of vals[0..n), n <= 64, by one warp; all lanes return it.
__device__ __forceinline__ float warp_kth_largest(const float* vals, int n, int k) {
  const int lane = threadIdx.x & 31;
  float res = -INFINITY;
  for (int g = lane; g < n; g += 32) {
    const float v = vals[g];
    int rank = 0;
    for (int q = 0; q < n; ++q) {
      const float w = vals[q];
      rank += (w > v) | ((w == v) & (q < g));
    }
    if (rank == k - 1) res = v;
  }
  return warp_max(res);  // exactly one lane holds it, the others hold -inf
}

__device__ __forceinline__ const float* rec_ptr(const StepParams& p, long long u) {
  return reinterpret_cast<const float*>(p.rec + (size_t)u * p.rec_stride);
}

__device__ __forceinline__ void write_output(const StepParams& p, const SelSmem& sm, int b, int r, const Key& key) {
  const int o = b * p.k + r;
  const int parent = key_parent(key);
  const int token = key_token(key);
  p.out_token[o] = token;
  p.out_parent[o] = parent;
  p.out_score[o] = key_score(key);
  if (p.out_finished) p.out_finished[o] = (sm.fin[parent] || token == p.eos) ? 1 : 0;
}

__device__ __forceinline__ void write_row_stats(const StepParams& p, const SelSmem& sm, int b, bool exact) {
  for (int j = threadIdx.x; j < p.k; j += kSelThreads) {
    const RowSel rs = sm.row[j];
    RowStat st;
    st.lse = rs.kind == ROW_FIN ? __int_as_float(0x7fc00000) : rs.lse;
    st.rtopk = rs.rtopk;
    st.ncand = exact ? -1 : rs.ncand;
    st.pad = 0;
    p.rowstat[b * p.k + j] = st;
  }
}

// Sort a[0..n) ascending by key (n a power of two); all threads call it.
__device__ void bitonic_sort(Key* a, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += kSelThreads) {
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
__device__ void merge_into_best(SelSmem& sm, int K) {
  const int nb = sm.nbest, nr = sm.nrl;
  const int tot = nb + nr;
  int n = 1;
  while (n < tot) n <<= 1;
  for (int i = threadIdx.x; i < n; i += kSelThreads) {
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
  for (int i = threadIdx.x; i < keep; i += kSelThreads) sm.best[i] = sm.mg[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    sm.nbest = keep;
    sm.nrl = 0;
  }
  __syncthreads();
}

// Exact fine rank of batch b without the candidate queue: per live beam its top-K entries
// (order: larger x first, then smaller token id), merged across beams.
//  1. One pass over the beam's source keeps the entries x >= R (the beam's R-top-k, never
//     above its K-th largest, so its top-K are among them) in a shared-memory list.  The
//     source is the beam's slots when they hold every entry at or above R -- the queue only
//     outgrew the fine rank (path 3), or there are no logits (the projection's epilogue wrote
//     the slots) -- and its row otherwise (a chunk's slots overflowed, or the exact path is
//     forced), read in 16-byte vectors.
//  2. The top-K of that list: by counting ranks when it is short, else by a radix select of
//     the K-th largest order key over it; entries equal to that key are taken by smallest
//     token.  A list longer than the buffer (massive ties at R) falls back to the radix
//     select over the whole source, in token order.
constexpr int kExactBuf = 4096;  // entries (x, token) of a beam's list in dynamic shared memory
constexpr int kExactRankMax = 256;  // lists up to this long are ranked by counting
constexpr int kExactWarpList = kExactBuf / kSelWarps;  // a warp's list in the beam-parallel form

__host__ __device__ constexpr int pow2_at_least(int x) {
  int n = 1;
  while (n < x) n <<= 1;
  return n;
}

// Dynamic shared memory of K2 for k: the exact path's lists, then k * k rank keys.
__host__ __device__ constexpr size_t exact_smem_bytes(int k) {
  return kExactBuf * sizeof(float2) + (size_t)pow2_at_least(k * k) * sizeof(Key);
}

static_assert(exact_smem_bytes(kMaxK) <= (size_t)kSelStageMax, "the exact path's shared memory exceeds K2's limit");

// A warp's full list of entries (x, token): the k-th largest x among list[0..n) (n >= k), the
// larger of it and R as the new bound, and the entries at or above that bound kept in order.
// Returns (bound, kept count as int bits).  Out of line: it is called from unrolled loops.
__device__ __noinline__ float2 list_tighten(float2* list, int n, int K, float R) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  float kth = -INFINITY;
  for (int i = lane; i < n; i += 32) {
    const float xi = list[i].x;
    int gt = 0, ge = 0;
    for (int q = 0; q < n; ++q) {
      const float xq = list[q].x;
      gt += xq > xi;
      ge += xq >= xi;
    }
    if (gt < K && ge >= K) kth = xi;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kth = fmaxf(kth, __shfl_xor_sync(0xffffffffu, kth, o));
  R = fmaxf(R, kth);
  int out = 0;
  for (int b0 = 0; b0 < n; b0 += 32) {
    const int i = b0 + lane;
    const float2 en = i < n ? list[i] : make_float2(-INFINITY, 0.0f);
    const bool keep = i < n && en.x >= R;
    const unsigned bm = __ballot_sync(0xffffffffu, keep);
    __syncwarp();
    if (keep) list[out + __popc(bm & lt_mask)] = en;
    out += __popc(bm);
    __syncwarp();
  }
  return make_float2(R, __int_as_float(out));
}

// The exact path one warp per beam: each warp keeps its beam's entries x >= R in its own list
// -- from the beam's slots when they are complete, else from its row in 16-byte vectors -- and
// ranks them, writing the beam's top-k as rank keys; the batch's top-k are then the first k of
// the k * k keys, sorted once.  Returns false, with nothing written, when some beam has more
// such entries than a warp's list holds.
template <int DT, bool BIAS>
__device__ bool exact_parallel(const StepParams& p, SelSmem& sm, int b, int path, unsigned char* dyn,
                               bool from_slots) {
  constexpr int ES = Traits<DT>::kBytes;
  constexpr int VEC = Traits<DT>::kVec;
  const int K = p.k, C = p.slot_cap, nc = p.nc, V = p.vocab;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  float2* list = reinterpret_cast<float2*>(dyn) + warp * kExactWarpList;
  Key* keys = reinterpret_cast<Key*>(dyn + kExactBuf * sizeof(float2));
  const int nk = pow2_at_least(K * K);
  Key pad;
  pad.hi = ~0ull;
  pad.lo = ~0ull;
  if (tid == 0) sm.big = 0;
  __syncthreads();
  for (int j = warp; j < K; j += kSelWarps) {
    const RowSel rs = sm.row[j];
    const int row = b * K + j;
    Key* out = keys + j * K;
    if (rs.kind == ROW_FIN) {
      for (int r = lane; r < K; r += 32) out[r] = r == 0 ? make_key(p.beam[row], j, 0.0f, p.eos) : pad;
      continue;
    }
    if (rs.kind == ROW_DEAD) {
      for (int r = lane; r < K; r += 32) out[r] = make_key(-INFINITY, j, 0.0f, r);
      continue;
    }
    float R = rs.rtopk;
    int n = 0;
    bool full = false;  // ties at the bound beyond the list: the serial path takes the batch
    // The list is full: raise R to the k-th largest of its entries (elements of the row, so
    // still a lower bound of its k-th largest) and keep the entries at or above it.
    auto tighten = [&]() {
      const float2 rn = list_tighten(list, n, K, R);
      R = rn.x;
      n = __float_as_int(rn.y);
    };
    auto append = [&](bool take, float x, int v) {
      unsigned m = __ballot_sync(0xffffffffu, take);
      if (n + __popc(m) > kExactWarpList) {
        tighten();
        m = __ballot_sync(0xffffffffu, take && x >= R);
        if (n + __popc(m) > kExactWarpList) {
          full = true;
          return;
        }
      }
      const int pos = n + __popc(m & lt_mask);
      if ((m >> lane) & 1u) list[pos] = make_float2(x, __int_as_float(v));
      n += __popc(m);
    };
    if (from_slots) {
      const long long u0 = (long long)row * nc;
      for (int c = 0; c < nc && !full; ++c) {
        const int cnt = min(__float_as_int(rec_ptr(p, u0 + c)[0]), C);
        const CandSlot* sl = p.slots + (u0 + c) * C;
        for (int s0 = 0; s0 < cnt; s0 += 32) {
          const int i = s0 + lane;
          CandSlot cs;
          cs.x = -INFINITY;
          cs.v = 0;
          if (i < cnt) cs = sl[i];
          append(i < cnt && cs.x >= R, cs.x, cs.v);
        }
      }
    } else {
      // 16-byte vectors covering the row (the first may start before it, the last end after
      // it), four per lane in flight
      const unsigned char* rowp = static_cast<const unsigned char*>(p.logits) + (size_t)row * V * ES;
      const int lead = (int)(reinterpret_cast<uintptr_t>(rowp) & 15);
      const uint4* rb = reinterpret_cast<const uint4*>(rowp - lead);
      const int row_bytes = V * ES;
      const int nv = (lead + row_bytes + 15) >> 4;
      for (int v0 = 0; v0 < nv && !full; v0 += 128) {
        uint4 d[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int jv = v0 + 32 * r + lane;
          d[r] = jv < nv ? __ldcs(rb + jv) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll 1
        for (int r = 0; r < 4; ++r) {
          const int jv = v0 + 32 * r + lane;
          float xs[VEC];
          const uint4 dv = r == 0 ? d[0] : (r == 1 ? d[1] : (r == 2 ? d[2] : d[3]));  // no local array
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
    }
    if (full) {
      if (lane == 0) sm.big = 1;
      continue;
    }
    __syncwarp();
    for (int r = n + lane; r < K; r += 32) out[r] = pad;  // fewer than k entries (cannot happen for a live beam)
    for (int i = lane; i < n; i += 32) {
      const float2 ei = list[i];
      const int vi = __float_as_int(ei.y);
      int rank = 0;
      for (int q = 0; q < n; ++q) {
        const float2 eq = list[q];
        rank += (eq.x > ei.x) | ((eq.x == ei.x) & (__float_as_int(eq.y) < vi));
      }
      if (rank < K) out[rank] = make_key(score_of(rs.c, ei.x), j, ei.x, vi);
    }
  }
  __syncthreads();
  if (sm.big) return false;
  for (int i = K * K + tid; i < nk; i += kSelThreads) keys[i] = pad;
  __syncthreads();
  bitonic_sort(keys, nk);
  for (int r = tid; r < K; r += kSelThreads) write_output(p, sm, b, r, keys[r]);
  write_row_stats(p, sm, b, true);
  if (tid == 0) p.bstat[b] = path;
  return true;
}

template <int DT, bool BIAS>
__device__ void exact_select(const StepParams& p, SelSmem& sm, int b, int path, float2* buf) {
  constexpr int ES = Traits<DT>::kBytes;
  constexpr int VEC = Traits<DT>::kVec;
  constexpr int NT = kSelThreads;
  const int K = p.k, V = p.vocab, C = p.slot_cap, nc = p.nc;
  const bool from_slots = p.logits == nullptr || path == 3;
  if (exact_parallel<DT, BIAS>(p, sm, b, path, reinterpret_cast<unsigned char*>(buf), from_slots)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
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
      for (int v = tid; v < K; v += NT) sm.rl[v] = make_key(-INFINITY, j, 0.0f, v);
      if (tid == 0) sm.nrl = K;
      __syncthreads();
      merge_into_best(sm, K);
      continue;
    }
    const unsigned char* rowp = p.logits ? static_cast<const unsigned char*>(p.logits) + (size_t)row * V * ES : nullptr;
    const long long u0 = (long long)row * nc;
    const int n_src = from_slots ? nc * C : V;
    // entry i of the beam's source, in token order: (x, token), or false when i is empty
    auto src = [&](int i, float& x, int& v) -> bool {
      if (from_slots) {
        const int c = i / C, sl = i - c * C;
        if (sl >= __float_as_int(rec_ptr(p, u0 + c)[0])) return false;
        const CandSlot cs = p.slots[(u0 + c) * C + sl];
        x = cs.x;
        v = cs.v;
        return true;
      }
      x = load_elem<DT>(rowp + (size_t)i * ES);
      if constexpr (BIAS) x += __ldg(p.bias + i);
      v = i;
      return true;
    };
    // 1. the entries at or above R, appended a warp at a time
    const float R = rs.rtopk;
    if (tid == 0) sm.ecnt = 0;
    __syncthreads();
    auto append = [&](bool take, float x, int v) {
      const unsigned m = __ballot_sync(0xffffffffu, take);
      if (m == 0u) return;
      int base = 0;
      if (lane == 0) base = atomicAdd(&sm.ecnt, __popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      const int pos = base + __popc(m & lt_mask);
      if (take && pos < kExactBuf) buf[pos] = make_float2(x, __int_as_float(v));
    };
    if (from_slots) {
      for (int i0 = warp * 32; i0 < n_src; i0 += NT) {
        float x = 0.0f;
        int v = 0;
        const int i = i0 + lane;
        const bool take = i < n_src && src(i, x, v) && x >= R;
        append(take, x, v);
      }
    } else {
      // 16-byte vectors covering the row (the first may start before it, the last end after
      // it), four per thread in flight
      const int lead = (int)(reinterpret_cast<uintptr_t>(rowp) & 15);
      const uint4* rb = reinterpret_cast<const uint4*>(rowp - lead);
      const int row_bytes = V * ES;
      const int nv = (lead + row_bytes + 15) >> 4;
      for (int v0 = warp * 128; v0 < nv; v0 += NT * 4) {
        uint4 d[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int jv = v0 + 32 * r + lane;
          d[r] = jv < nv ? __ldcs(rb + jv) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll 1
        for (int r = 0; r < 4; ++r) {
          const int jv = v0 + 32 * r + lane;
          float xs[VEC];
          const uint4 dv = r == 0 ? d[0] : (r == 1 ? d[1] : (r == 2 ? d[2] : d[3]));  // no local array
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
    }
    __syncthreads();
    const int n = sm.ecnt;
    if (tid == 0) sm.nrl = 0;
    __syncthreads();
    if (n <= kExactRankMax) {
      // 2a. short list: each entry's rank among the others
      for (int i = tid; i < n; i += NT) {
        const float2 ei = buf[i];
        const int vi = __float_as_int(ei.y);
        int rank = 0;
        for (int q = 0; q < n; ++q) {
          const float2 eq = buf[q];
          const int vq = __float_as_int(eq.y);
          rank += (eq.x > ei.x) | ((eq.x == ei.x) & (vq < vi));
        }
        if (rank < K) sm.rl[rank] = make_key(score_of(rs.c, ei.x), j, ei.x, vi);
      }
      if (tid == 0) sm.nrl = n < K ? n : K;
    } else {
      // 2b. radix select of the K-th largest order key, 8 bits at a time from the top, over
      // the list (n <= kExactBuf) or, when it overflowed, over the whole source
      const bool over_buf = n <= kExactBuf;
      const int n_sel = over_buf ? n : n_src;
      auto entry = [&](int i, float& x, int& v) -> bool {
        if (over_buf) {
          const float2 e = buf[i];
          x = e.x;
          v = __float_as_int(e.y);
          return true;
        }
        return src(i, x, v);
      };
      if (tid == 0) {
        sm.prefix = 0;
        sm.pmask = 0;
        sm.need = K;
      }
      __syncthreads();
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += NT) sm.hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = sm.prefix, pmask = sm.pmask;
        for (int i = tid; i < n_sel; i += NT) {
          float x;
          int v;
          if (!entry(i, x, v)) continue;
          const uint32_t o = float_ord(x);
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
      const int need_eq = sm.need;  // entries equal to the threshold to take, smallest tokens first
      for (int i = tid; i < n_sel; i += NT) {
        float x;
        int v;
        if (!entry(i, x, v)) continue;
        if (float_ord(x) > tkey) {
          const int pos = atomicAdd(&sm.nrl, 1);
          if (pos < kMaxK) sm.rl[pos] = make_key(score_of(rs.c, x), j, x, v);
        }
      }
      __syncthreads();
      if (over_buf) {
        // the list is in no particular order: an equal entry is taken when fewer than need_eq
        // equal entries have a smaller token
        for (int i = tid; i < n_sel; i += NT) {
          const float2 ei = buf[i];
          if (float_ord(ei.x) != tkey) continue;
          const int vi = __float_as_int(ei.y);
          int before = 0;
          for (int q = 0; q < n_sel; ++q) {
            const float2 eq = buf[q];
            before += (float_ord(eq.x) == tkey) & (__float_as_int(eq.y) < vi);
          }
          if (before < need_eq) {
            const int pos = atomicAdd(&sm.nrl, 1);
            if (pos < kMaxK) sm.rl[pos] = make_key(score_of(rs.c, ei.x), j, ei.x, vi);
          }
        }
      } else {
        // the source is in token order: the first need_eq equal entries
        int taken = 0;
        for (int base = 0; base < n_sel && taken < need_eq; base += NT) {
          const int i = base + tid;
          float x = 0.0f;
          int v = 0;
          bool eq = false;
          if (i < n_sel && entry(i, x, v)) eq = float_ord(x) == tkey;
          const unsigned ballot = __ballot_sync(0xffffffffu, eq);
          if (lane == 0) sm.wc[warp] = __popc(ballot);
          __syncthreads();
          int before = 0, total = 0;
          for (int w = 0; w < kSelWarps; ++w) {
            before += (w < warp) ? sm.wc[w] : 0;
            total += sm.wc[w];
          }
          const int off = taken + before + __popc(ballot & lt_mask);
          if (eq && off < need_eq) {
            const int pos = atomicAdd(&sm.nrl, 1);
            if (pos < kMaxK) sm.rl[pos] = make_key(score_of(rs.c, x), j, x, v);
          }
          taken += total;
          __syncthreads();
        }
      }
      __syncthreads();
      if (tid == 0 && sm.nrl > kMaxK) sm.nrl = kMaxK;  // greater + taken equal == K, cannot exceed
    }
    __syncthreads();
    merge_into_best(sm, K);
  }
  for (int r = tid; r < K && r < sm.nbest; r += NT) write_output(p, sm, b, r, sm.best[r]);
  write_row_stats(p, sm, b, true);
  if (tid == 0) p.bstat[b] = path;
}

// Fine rank of batch b for k <= 8 (G <= 8 group maxima per beam) with at most 128 chunks per
// beam and kPairTile (beam, chunk) pairs per batch: the common case, kept short because the
// code runs once per CTA right after K1 (every instruction line is fetched cold).
//   AB. warp j merges beam j's chunk records (loads issued together): the row max M, then
//       S = sum of the chunk sums rescaled to M, the G group maxima and the row-level
//       R-top-k (k-th largest of them); lse = M + log S.
//   C.  each warp flattens the slots of its own run of pairs (a warp scan, no CTA barrier),
//       keeps the slots with x >= R of their beam and rescores them into rank keys.
//   D.  each key's rank is counted against the others; ranks < k are the outputs.
// Returns the path: 0 when the outputs are written, otherwise the reason for the exact path.
//
// With dry = true the same code runs without any global store and with its loops capped,
// on whatever the workspace holds: a CTA that becomes resident while K1 is still running
// makes this pass before waiting on K1, so that the instructions of the real pass are
// already in the SM's instruction cache (fetching them cold costs microseconds per phase,
// more than the work itself).  Every count and address stays clamped, so stale or
// half-written records are harmless; nothing the dry pass computes is kept.
template <int DT, bool BIAS>
__device__ __forceinline__ int queue_select(const StepParams& p, SelSmem& sm, unsigned char* stage, int b, bool dry) {
  const int K = p.k, nc = p.nc, G = p.groups, C = p.slot_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long ub = (long long)b * K * nc;
  // the batch's slots (contiguous) land in shared memory while AB runs
  const bool staged = !dry && p.sel_stage_bytes > 0;
  if (staged && tid == 0) {
    const uint32_t bar = smem_addr(&sm.sbar);
    mbar_init(bar, 1);
    fence_barrier_init();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    mbar_arrive_expect_tx(bar, (uint32_t)p.sel_stage_bytes);
    bulk_load_plain(smem_addr(stage), p.slots + (size_t)ub * C, (uint32_t)p.sel_stage_bytes, bar);
  }
  // AB
  if (warp < K) {
    const int j = warp;
    if (sm.fin[j]) {
      if (lane == 0) {
        RowSel rs;
        rs.c = ScoreBase{0.0f, 0.0f};
        rs.rtopk = __int_as_float(0x7fc00000);
        rs.lse = __int_as_float(0x7fc00000);
        rs.kind = ROW_FIN;
        rs.ncand = 1;
        sm.row[j] = rs;
      }
    } else {
      const long long u0 = ((long long)b * K + j) * nc;
      float m[4], sc[4];
      float4 ga[4], gb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        m[i] = -INFINITY;
        sc[i] = 0.0f;
        ga[i] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        gb[i] = ga[i];
        if (c < nc) {
          const float4* r4 = reinterpret_cast<const float4*>(rec_ptr(p, u0 + c));
          const float4 h = __ldcg(r4);
          ga[i] = __ldcg(r4 + 1);
          if (G > 4) gb[i] = __ldcg(r4 + 2);
          m[i] = h.y;
          sc[i] = h.z;
          sm.pn[j * nc + c] = dry ? 0 : __float_as_int(h.x);
        }
      }
      const float M = warp_max(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])));
      float ls = 0.0f;
      bool ovf = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        if (c < nc) {
          if (m[i] != -INFINITY) ls += sc[i] * exp2f((m[i] - M) * kLog2e);
          sm.pm[j * nc + c] = m[i];
          ovf |= sm.pn[j * nc + c] > C;
        }
      }
      float S = ls;
#pragma unroll 1
      for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
      // group maxima: lane-local over its chunks, then over the warp
      float g8[8] = {ga[0].x, ga[0].y, ga[0].z, ga[0].w, gb[0].x, gb[0].y, gb[0].z, gb[0].w};
#pragma unroll
      for (int i = 1; i < 4; ++i) {
        g8[0] = fmaxf(g8[0], ga[i].x);
        g8[1] = fmaxf(g8[1], ga[i].y);
        g8[2] = fmaxf(g8[2], ga[i].z);
        g8[3] = fmaxf(g8[3], ga[i].w);
        g8[4] = fmaxf(g8[4], gb[i].x);
        g8[5] = fmaxf(g8[5], gb[i].y);
        g8[6] = fmaxf(g8[6], gb[i].z);
        g8[7] = fmaxf(g8[7], gb[i].w);
      }
#pragma unroll 1
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int g = 0; g < 8; ++g) g8[g] = fmaxf(g8[g], __shfl_xor_sync(0xffffffffu, g8[g], o));
      }
      // every lane holds the G group maxima; R = the k-th largest of them
      float R = g8[0];
      if (G == K) {
        // k group maxima: the k-th largest is the least one
#pragma unroll
        for (int g = 1; g < 8; ++g) R = g < G ? fminf(R, g8[g]) : R;
      } else {
        // lane g < G takes group max g and counts the larger ones (ties by group index)
        float v = g8[0];
#pragma unroll
        for (int g = 1; g < 8; ++g) v = lane == g ? g8[g] : v;
        int rank = 0;
#pragma unroll 1
        for (int q = 0; q < G; ++q) {
          const float w = __shfl_sync(0xffffffffu, v, q);
          rank += (w > v) | ((w == v) & (q < lane));
        }
        const unsigned hit = __ballot_sync(0xffffffffu, lane < G && rank == K - 1);
        R = __shfl_sync(0xffffffffu, v, __ffs(hit) - 1);
      }
      ovf = __any_sync(0xffffffffu, ovf);
      if (lane == 0) {
        const float beam = sm.beam[j];
        RowSel rs;
        rs.rtopk = R;
        rs.ncand = 0;
        if (M == -INFINITY || beam == -INFINITY) {
          rs.kind = ROW_DEAD;
          rs.c = ScoreBase{-INFINITY, 0.0f};
          rs.lse = M == -INFINITY ? -INFINITY : M + logf(S);
        } else {
          const float log_s = logf(S);
          rs.kind = ROW_LIVE;
          rs.c = score_base(beam, M, log_s);  // beam - lse, lse = M + log S
          rs.lse = __fadd_rn(M, log_s);
        }
        sm.row[j] = rs;
        if (ovf) sm.ovf = 1;
      }
    }
  }
  __syncthreads();
  if (!dry) {
    if (sm.ovf) return 1;
    if (p.flags & kFlagForceExact) return 2;
  }

  // C: warp w takes pairs [qb, qe); pair q = j * nc + c
  const int P = K * nc;
  const int T = (P + kSelWarps - 1) / kSelWarps;
  const int qb = warp * T, qe = min(P, qb + T);
  int run = 0;
#pragma unroll 1
  for (int q0 = qb; q0 < qe; q0 += 32) {
    const int q = q0 + lane;
    int cnt = 0;
    if (q < qe) {
      const RowSel& rs = sm.row[q / nc];
      if (dry)
        cnt = 1;  // one slot per pair: every load below stays inside the pair's slots
      else if (rs.kind == ROW_LIVE && sm.pm[q] >= rs.rtopk)
        cnt = min(sm.pn[q], C);
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (q < qe) sm.pc[q] = run + incl - cnt;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  if (staged && !mbar_wait_bounded(smem_addr(&sm.sbar), 0, p.spin_limit_ns)) {
    // the copy did not complete in time: record it, let it land, write nothing
    if (tid == 0) {
      atomicOr(p.status, kDevTimeout);
      mbar_wait_bounded(smem_addr(&sm.sbar), 0, 2000000000LL);
    }
    __syncthreads();
    return -1;
  }
  if (dry) run = min(run, 32);
  const CandSlot* sslots = reinterpret_cast<const CandSlot*>(stage);
  const unsigned lt_mask = (1u << lane) - 1u;
  // 4 slots per lane per round, loads issued together; no data-dependent branch (a
  // divergent branch costs more than the work it guards here)
  // binary-search depth: the largest power of two below the warp's pair count
  int top = 1;
  while (top * 2 < qe - qb) top *= 2;
#pragma unroll 1
  for (int i0 = 0; i0 < run; i0 += 4 * 32) {
    int2 raw[4];
    int jj[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int i = i0 + t * 32 + lane;
      jj[t] = -1;
      raw[t] = make_int2((int)0xff800000u, 0);
      if (i0 + t * 32 < run) {  // warp-uniform
        // last pair of [qb, qe) whose prefix is <= i
        int lo = qb;
#pragma unroll 1
        for (int st = top; st > 0; st >>= 1) {
          const int cand = min(lo + st, qe - 1);
          lo = (sm.pc[cand] <= i) ? cand : lo;
        }
        if (i < run) {
          jj[t] = (int)fast_div((uint32_t)lo, p.nc_magic, p.nc_shift);
          const size_t si = (size_t)lo * C + (i - sm.pc[lo]);
          raw[t] = staged ? *reinterpret_cast<const int2*>(sslots + si)
                          : __ldcg(reinterpret_cast<const int2*>(p.slots + (size_t)ub * C + si));
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int jr = max(jj[t], 0);
      const float x = __int_as_float(raw[t].x);
      const RowSel& rs = sm.row[jr];
      const bool surv = (jj[t] >= 0) & (x >= rs.rtopk);
      const unsigned m = __ballot_sync(0xffffffffu, surv);
      if (m != 0u) {  // warp-uniform
        int base = 0;
        if (lane == 0) base = atomicAdd(&sm.nsel, __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(m & lt_mask);
        if (surv & (pos < kSelCap)) sm.sel[pos] = make_key(score_of(rs.c, x), jr, x, raw[t].y);
        // survivors per beam: the first lane of each beam's group adds the group's count
        const unsigned same = __match_any_sync(0xffffffffu, surv ? jr : -1);
        if (surv & ((same & lt_mask) == 0u)) atomicAdd(&sm.row[jr].ncand, __popc(same));
      }
    }
  }
  // finished beams offer (eos_id, beam score); beams with no finite score offer k tokens
  if (tid < K * K) {
    const int jr = tid / K, v = tid - jr * K;
    const int kind = sm.row[jr].kind;
    if ((kind == ROW_FIN && v == 0) || kind == ROW_DEAD) {
      const int pos = atomicAdd(&sm.nsel, 1);
      if (pos < kSelCap)
        sm.sel[pos] = kind == ROW_FIN ? make_key(sm.beam[jr], jr, 0.0f, p.eos) : make_key(-INFINITY, jr, 0.0f, v);
      else
        sm.big = 1;
      if (kind == ROW_DEAD && v == 0) sm.row[jr].ncand = K;
    }
  }
  __syncthreads();
  if ((sm.big || sm.nsel > kSelCap) && !dry) return 3;
  // D
  const int n = dry ? min(sm.nsel, 32) : sm.nsel;
#pragma unroll 1
  for (int i = tid; i < n; i += kSelThreads) {
    const Key ki = sm.sel[i];
    int r0 = 0, r1 = 0;
    int q = 0;
#pragma unroll 1
    for (; q + 1 < n; q += 2) {
      r0 += key_less(sm.sel[q], ki);
      r1 += key_less(sm.sel[q + 1], ki);
    }
    if (q < n) r0 += key_less(sm.sel[q], ki);
    if (r0 + r1 < K && !dry) write_output(p, sm, b, r0 + r1, ki);
  }
  if (!dry) {
    write_row_stats(p, sm, b, false);
    if (tid == 0) p.bstat[b] = 0;
  }
  return 0;
}

template <int DT, bool BIAS>
__global__ void __launch_bounds__(kSelThreads, 1) beam_select_kernel(const StepParams p) {
  __shared__ SelSmem sm;
  extern __shared__ __align__(128) unsigned char sel_stage[];
  const int K = p.k, nc = p.nc, G = p.groups, C = p.slot_cap;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  if (tid == 0) {
    sm.nsel = 0;
    sm.big = 0;
    sm.ovf = 0;
  }
  // inputs that do not come from K1: read before waiting on it
  for (int j = tid; j < K; j += kSelThreads) {
    sm.beam[j] = p.beam[b * K + j];
    sm.fin[j] = (p.finished && p.finished[b * K + j]) ? 1 : 0;
  }
  __syncthreads();
  const bool queue_path = K <= 8 && nc <= 128 && K * nc <= kPairTile;
  if (queue_path) {
    queue_select<DT, BIAS>(p, sm, sel_stage, b, true);  // warms the instruction cache (no stores)
    __syncthreads();
    if (tid == 0) {
      sm.nsel = 0;
      sm.big = 0;
      sm.ovf = 0;
    }
  }
  grid_dependency_wait();  // K1's records and slots are complete and visible
  __syncthreads();
  if (queue_path) {
    const int path = queue_select<DT, BIAS>(p, sm, sel_stage, b, false);
    if (path > 0) exact_select<DT, BIAS>(p, sm, b, path, reinterpret_cast<float2*>(sel_stage));
    return;
  }
  const bool keep_pairs = K * nc <= kPairTile;
  // 1. per beam: log_sum_exp, the row-level R-top-k and the score offset
  for (int j = warp; j < K; j += kSelWarps) {
    const bool fin = sm.fin[j] != 0;
    const float beam = sm.beam[j];
    if (fin) {
      if (lane == 0) {
        RowSel rs;
        rs.c = ScoreBase{0.0f, 0.0f};
        rs.rtopk = __int_as_float(0x7fc00000);
        rs.lse = __int_as_float(0x7fc00000);
        rs.kind = ROW_FIN;
        rs.ncand = 1;
        sm.row[j] = rs;
      }
      continue;
    }
    const long long u0 = (long long)(b * K + j) * nc;
    // one pass over the chunk records: (max, sum of exp) with online rescaling, the group
    // maxima (G <= 8 held per lane), then fixed shuffle trees (deterministic)
    float M = -INFINITY, S = 0.0f;
    bool ovf = false;
    float gl[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) gl[g] = -INFINITY;
    for (int c = lane; c < nc; c += 32) {
      const float4* r4 = reinterpret_cast<const float4*>(rec_ptr(p, u0 + c));
      const float4 h = r4[0];
      float4 ga = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY), gb = ga;
      if (G <= 8) {
        ga = r4[1];
        if (G > 4) gb = r4[2];
      }
      const int cnt = __float_as_int(h.x);
      const float mc = h.y, sc = h.z;
      if (keep_pairs) {
        sm.pm[j * nc + c] = mc;
        sm.pn[j * nc + c] = cnt;
      }
      ovf |= cnt > C;
      const float Mn = fmaxf(M, mc);
      if (Mn != -INFINITY) {
        S = (M == -INFINITY ? 0.0f : S * exp2f((M - Mn) * kLog2e)) +
            (mc == -INFINITY ? 0.0f : sc * exp2f((mc - Mn) * kLog2e));
        M = Mn;
      }
      gl[0] = fmaxf(gl[0], ga.x);
      gl[1] = fmaxf(gl[1], ga.y);
      gl[2] = fmaxf(gl[2], ga.z);
      gl[3] = fmaxf(gl[3], ga.w);
      gl[4] = fmaxf(gl[4], gb.x);
      gl[5] = fmaxf(gl[5], gb.y);
      gl[6] = fmaxf(gl[6], gb.z);
      gl[7] = fmaxf(gl[7], gb.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
      const float So = __shfl_xor_sync(0xffffffffu, S, o);
      const float Mn = fmaxf(M, Mo);
      if (Mn != -INFINITY) {
        S = (M == -INFINITY ? 0.0f : S * exp2f((M - Mn) * kLog2e)) +
            (Mo == -INFINITY ? 0.0f : So * exp2f((Mo - Mn) * kLog2e));
      }
      M = Mn;
    }
    ovf = __any_sync(0xffffffffu, ovf);
    if (G <= 8) {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float v = warp_max(gl[g]);
        if (lane == 0 && g < G) sm.selg[warp][g] = v;
      }
    } else if (G <= 32) {
      // group maxima merged over the chunks: lanes split the (chunk, group) pairs
      const int g = lane & (G - 1);
      const int cs = 32 / G;
      float gm = -INFINITY;
      for (int c0 = lane / G; c0 < nc; c0 += 4 * cs) {
        float v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int c = c0 + t * cs;
          v[t] = c < nc ? rec_ptr(p, u0 + c)[4 + g] : -INFINITY;
        }
        gm = fmaxf(gm, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
      }
      for (int o = 16; o >= G; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
      if (lane < G) sm.selg[warp][lane] = gm;
    } else {
      float ga = -INFINITY, gb = -INFINITY;
      for (int c = 0; c < nc; ++c) {
        const float* r = rec_ptr(p, u0 + c);
        ga = fmaxf(ga, r[4 + lane]);
        gb = fmaxf(gb, r[4 + 32 + lane]);
      }
      sm.selg[warp][lane] = ga;
      sm.selg[warp][32 + lane] = gb;
    }
    __syncwarp();
    const float rt = warp_kth_largest(sm.selg[warp], G, K);
    if (lane == 0) {
      RowSel rs;
      rs.rtopk = rt;
      rs.ncand = 0;
      if (M == -INFINITY || beam == -INFINITY) {
        rs.kind = ROW_DEAD;
        rs.c = ScoreBase{-INFINITY, 0.0f};
        rs.lse = M == -INFINITY ? -INFINITY : M + logf(S);
      } else {
        const float log_s = logf(S);
        rs.kind = ROW_LIVE;
        rs.c = score_base(beam, M, log_s);  // beam - lse, lse = M + log S
        rs.lse = __fadd_rn(M, log_s);
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
    // 2. survivors of the row-level R-top-k, rescored: beam_score + x - lse.  The slots of
    // all (beam, chunk) pairs are flattened so that every load is independent.
    const int P = K * nc;
    for (int t0 = 0; t0 < P; t0 += kPairTile) {
      const int nt = min(kPairTile, P - t0);
      for (int i = tid; i < nt; i += kSelThreads) {
        const int pair = t0 + i;
        const int j = pair / nc;
        int c = 0;
        if (sm.row[j].kind == ROW_LIVE) {
          // a chunk whose max is below the beam's R-top-k holds no survivor: skip its slots
          float mc;
          int n;
          if (keep_pairs) {
            mc = sm.pm[pair];
            n = sm.pn[pair];
          } else {
            const float* r = rec_ptr(p, (long long)b * K * nc + pair);
            mc = r[1];
            n = reinterpret_cast<const int*>(r)[0];
          }
          if (mc >= sm.row[j].rtopk) c = min(n, C);
        }
        sm.pc[i] = c;
      }
      __syncthreads();
      // exclusive scan of pc[0..nt): 4 consecutive entries per thread
      constexpr int kPer = kPairTile / kSelThreads;
      int loc[kPer];
      int run = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        const int i = tid * kPer + e;
        loc[e] = run;
        run += (i < nt) ? sm.pc[i] : 0;
      }
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) sm.wsum[warp] = incl;
      __syncthreads();
      int wbase = 0, tot = 0;
      for (int w = 0; w < kSelWarps; ++w) {
        wbase += (w < warp) ? sm.wsum[w] : 0;
        tot += sm.wsum[w];
      }
      const int tbase = wbase + incl - run;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        const int i = tid * kPer + e;
        if (i < nt) sm.pc[i] = tbase + loc[e];
      }
      __syncthreads();
      // 4 slots per thread per round, their loads issued together
      for (int q0 = tid; q0 < tot; q0 += 4 * kSelThreads) {
        int2 raw[4];
        int jj[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int q = q0 + t * kSelThreads;
          jj[t] = -1;
          if (q < tot) {
            int lo = 0, hi = nt - 1;  // last pair with prefix <= q
            while (lo < hi) {
              const int mid = (lo + hi + 1) >> 1;
              if (sm.pc[mid] <= q)
                lo = mid;
              else
                hi = mid - 1;
            }
            const int pair = t0 + lo;
            jj[t] = pair / nc;
            const long long u = (long long)b * K * nc + pair;
            raw[t] = *reinterpret_cast<const int2*>(p.slots + (size_t)u * C + (q - sm.pc[lo]));
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (jj[t] < 0) continue;
          const int j = jj[t];
          const float x = __int_as_float(raw[t].x);
          const RowSel& rs = sm.row[j];
          if (x >= rs.rtopk) {
            const Key key = make_key(score_of(rs.c, x), j, x, raw[t].y);
            const int pos = atomicAdd(&sm.nsel, 1);
            if (pos < kSelCap)
              sm.sel[pos] = key;
            else
              sm.big = 1;
            atomicAdd(&sm.row[j].ncand, 1);
          }
        }
      }
      __syncthreads();
    }
    for (int idx = tid; idx < K * K; idx += kSelThreads) {
      const int j = idx / K, v = idx - (idx / K) * K;
      const int kind = sm.row[j].kind;
      if (kind == ROW_FIN && v == 0) {
        const int pos = atomicAdd(&sm.nsel, 1);
        if (pos < kSelCap)
          sm.sel[pos] = make_key(sm.beam[j], j, 0.0f, p.eos);
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
    exact_select<DT, BIAS>(p, sm, b, path, reinterpret_cast<float2*>(sel_stage));
    return;
  }
  // 3. rank of every survivor among the survivors; ranks 0..K-1 are the output
  const int n = sm.nsel;
  for (int i = tid; i < n; i += kSelThreads) {
    const Key ki = sm.sel[i];
    int rank = 0;
    for (int q = 0; q < n; ++q) rank += key_less(sm.sel[q], ki);
    if (rank < K) write_output(p, sm, b, rank, ki);
  }
  write_row_stats(p, sm, b, false);
  if (tid == 0) p.bstat[b] = 0;
}

template <int DT, bool BIAS>
cudaError_t launch_t(const StepParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.batch);
  cfg.blockDim = dim3(kSelThreads);
  // the slots' staging copy, or the exact path's list (the two are never in use at once)
  const size_t exact_bytes = exact_smem_bytes(p.k);
  cfg.dynamicSmemBytes = (size_t)p.sel_stage_bytes > exact_bytes ? (size_t)p.sel_stage_bytes : exact_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, beam_select_kernel<DT, BIAS>, p);
}

template <int DT, bool BIAS>
cudaError_t config_t() {
  return cudaFuncSetAttribute(beam_select_kernel<DT, BIAS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelStageMax);
}

}  // namespace

cudaError_t beam_select_config() {
  cudaError_t e = config_t<DT_F32, false>();
  if (e == cudaSuccess) e = config_t<DT_F32, true>();
  if (e == cudaSuccess) e = config_t<DT_F16, false>();
  if (e == cudaSuccess) e = config_t<DT_F16, true>();
  if (e == cudaSuccess) e = config_t<DT_BF16, false>();
  if (e == cudaSuccess) e = config_t<DT_BF16, true>();
  return e;
}

cudaError_t launch_beam_select(const StepParams& p, int dtype, cudaStream_t stream) {
  const bool bias = p.bias != nullptr;
  switch (dtype) {
    case DT_F32: return bias ? launch_t<DT_F32, true>(p, stream) : launch_t<DT_F32, false>(p, stream);
    case DT_F16: return bias ? launch_t<DT_F16, true>(p, stream) : launch_t<DT_F16, false>(p, stream);
    case DT_BF16: return bias ? launch_t<DT_BF16, true>(p, stream) : launch_t<DT_BF16, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsb
