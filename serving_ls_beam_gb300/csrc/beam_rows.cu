// Beam-step kernel K1: the first and second traversal of every beam's logits, one
// chunk at a time, each chunk owned by a single warp.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), hierarchical decoding
// section.  First traversal: split a beam's logits into k groups, take each group's
// max; the k-th largest of those maxima (their min when there are exactly k groups)
// is the R-top-k bound, never above the true k-th largest; log_sum_exp in the same
// pass.  Second traversal: keep the logits at or above R-top-k as candidates.
//
// GB300 design:
//  * Work unit = one chunk of 32 x VPL 16-byte vectors of one beam's row.  Every warp
//    is an independent pipeline: lane 0 keeps a two-stage shared-memory ring full with
//    1-D bulk (TMA) copies completed on per-warp mbarriers, the warp reads the chunk
//    into registers and works on it while the next chunk lands.  No CTA barrier, no
//    fence and no global atomic on the streaming path; the logits are read from HBM
//    exactly once (L2 evict-first).
//  * Row boundaries need not be 16-byte aligned: a chunk is copied as whole aligned
//    vectors and the bytes outside the row are masked to -inf.
//  * Per chunk: (max, sum of exp) and the group maxima (group = lane mod G, G = the
//    power of two >= k; with G = 64 the two halves of a lane's vectors are two groups)
//    by warp shuffles; R-top-k of the chunk = k-th largest group max.  Any element of
//    the row's top-k lying in the chunk is in the chunk's own top-k, hence >= the
//    chunk's R-top-k, so the chunk's survivors can be taken before the row is complete.
//    They go to the chunk's own slot range (the batch's "queue" is the set of its
//    chunks' ranges), so no atomics are needed; a chunk with more survivors than slots
//    tightens its bound to the k-th largest of its 32 per-lane maxima and filters again.
//  * The chunk record (count, max, sum, group maxima) lets the fine-rank kernel rebuild
//    each beam's log_sum_exp and its row-level R-top-k (the article's k-group bound).
#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"

namespace lsb {
namespace {

// stages of a warp's ring: two for chunks up to 4 KB, one for 8 KB chunks (the other warps
// of the SM hide the load latency; the shared memory per warp stays 8 KB)
__host__ __device__ constexpr int stages_for(int vpl) { return vpl >= 16 ? 1 : 2; }
constexpr int kStagesMax = 2;
constexpr long long kDrainLimitNs = 2000000000LL;  // 2 s for copies already in flight
// shared-memory layout: [mbarriers | per-warp item lists | stage buffers]
static_assert(kRowWarps * kStagesMax * 8 <= kRowListOff, "mbarriers overlap the item lists");
static_assert(kRowBarBytes % 16 == 0, "stage buffers must be 16-byte aligned for bulk copies");

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// k-th largest (1-based) of the values held by lanes [0, n), n <= 32; all lanes get it.
__device__ __forceinline__ float warp_kth_of_lanes(float v, int n, int k) {
  const int lane = threadIdx.x & 31;
  int rank = 0;
  for (int q = 0; q < n; ++q) {
    const float w = __shfl_sync(0xffffffffu, v, q);
    rank += (w > v) | ((w == v) & (q < lane));
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < n && rank == k - 1);
  return __shfl_sync(0xffffffffu, v, __ffs(hit) - 1);
}

// k-th largest of 64 values, a = group lane, b = group lane + 32; all lanes get it.
__device__ __forceinline__ float warp_kth_of_64(float a, float b, int k) {
  const int lane = threadIdx.x & 31;
  int ra = 0, rb = 0;
  for (int q = 0; q < 32; ++q) {
    const float wa = __shfl_sync(0xffffffffu, a, q);
    const float wb = __shfl_sync(0xffffffffu, b, q);
    ra += (wa > a) | ((wa == a) & (q < lane));
    ra += (wb > a);
    rb += (wa >= b);
    rb += (wb > b) | ((wb == b) & (q < lane));
  }
  const bool ha = ra == k - 1, hb = rb == k - 1;
  const unsigned hit = __ballot_sync(0xffffffffu, ha || hb);
  const float mine = ha ? a : b;
  return __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1);
}

// Packed per-vector max: for 16-bit types a pair (max of even, max of odd elements) as
// the type's 2-vector, kept as its 32-bit pattern; for fp32 the max itself.
template <int DT>
__device__ __forceinline__ uint32_t vec_max_bits(const uint4& d) {
  if constexpr (DT == DT_F32) {
    return __float_as_uint(
        fmaxf(fmaxf(__uint_as_float(d.x), __uint_as_float(d.y)), fmaxf(__uint_as_float(d.z), __uint_as_float(d.w))));
  } else if constexpr (DT == DT_F16) {
    const __half2* h = reinterpret_cast<const __half2*>(&d);
    const __half2 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&d);
    const __nv_bfloat162 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return *reinterpret_cast<const uint32_t*>(&m);
  }
}
template <int DT>
__device__ __forceinline__ uint32_t max_bits(uint32_t a, uint32_t b) {
  if constexpr (DT == DT_F32) {
    return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
  } else if constexpr (DT == DT_F16) {
    const __half2 m = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __nv_bfloat162 m =
        __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  }
}
template <int DT>
__device__ __forceinline__ float bits_max_float(uint32_t a) {
  if constexpr (DT == DT_F32) {
    return __uint_as_float(a);
  } else if constexpr (DT == DT_F16) {
    const __half2 h = *reinterpret_cast<const __half2*>(&a);
    return fmaxf(__low2float(h), __high2float(h));
  } else {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&a);
    return fmaxf(__low2float(h), __high2float(h));
  }
}
// thr in the packed layout of type T (both halves for 16-bit types; thr is an element
// value, hence exact in the type)
template <int T>
__device__ __forceinline__ uint32_t thr_bits(float thr) {
  if constexpr (T == DT_F32) {
    return __float_as_uint(thr);
  } else if constexpr (T == DT_F16) {
    const __half2 t = __float2half2_rn(thr);
    return *reinterpret_cast<const uint32_t*>(&t);
  } else {
    const __nv_bfloat162 t = __float2bfloat162_rn(thr);
    return *reinterpret_cast<const uint32_t*>(&t);
  }
}
// true when either packed value reaches the packed threshold
template <int T>
__device__ __forceinline__ bool packed_ge(uint32_t a, uint32_t t) {
  if constexpr (T == DT_F32) {
    return __uint_as_float(a) >= __uint_as_float(t);
  } else if constexpr (T == DT_F16) {
    return __hge2_mask(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&t)) != 0u;
  } else {
    return __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&t)) != 0u;
  }
}

// Bit e set when element e of the vector is >= thr (values before any bias; thr is an
// element value, hence exact in the element type).
template <int DT>
__device__ __forceinline__ uint32_t vec_ge_mask(const uint4& d, float thr) {
  if constexpr (DT == DT_F32) {
    return (__uint_as_float(d.x) >= thr ? 1u : 0u) | (__uint_as_float(d.y) >= thr ? 2u : 0u) |
           (__uint_as_float(d.z) >= thr ? 4u : 0u) | (__uint_as_float(d.w) >= thr ? 8u : 0u);
  } else {
    const uint32_t t = thr_bits<DT>(thr);
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t g;
      if constexpr (DT == DT_F16) {
        g = __hge2_mask(*reinterpret_cast<const __half2*>(&w[i]), *reinterpret_cast<const __half2*>(&t));
      } else {
        g = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[i]), *reinterpret_cast<const __nv_bfloat162*>(&t));
      }
      m |= ((g & 1u) | ((g >> 15) & 2u)) << (2 * i);
    }
    return m;
  }
}

// Element e (runtime index) of a 16-byte vector as float, without dynamic register indexing.
template <int DT>
__device__ __forceinline__ float vec_elem(const uint4& d, int e) {
  if constexpr (DT == DT_F32) {
    const uint32_t w = e == 0 ? d.x : e == 1 ? d.y : e == 2 ? d.z : d.w;
    return __uint_as_float(w);
  } else {
    const int i = e >> 1;
    const uint32_t w = i == 0 ? d.x : i == 1 ? d.y : i == 2 ? d.z : d.w;
    const unsigned short h = (unsigned short)((e & 1) ? (w >> 16) : (w & 0xffffu));
    if constexpr (DT == DT_F16) {
      return __half2float(__ushort_as_half(h));
    } else {
      return __bfloat162float(__ushort_as_bfloat16(h));
    }
  }
}

template <int DT, bool BIAS, int VPL>
__global__ void __launch_bounds__(kRowThreads, VPL >= 16 ? 2 : 3) beam_rows_kernel(const StepParams p) {
  constexpr int kStages = stages_for(VPL);
  constexpr int VEC = Traits<DT>::kVec;
  constexpr int ES = Traits<DT>::kBytes;
  constexpr int CV = 32 * VPL;  // vectors per chunk
  constexpr uint32_t kStageBytes = CV * 16;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem_raw) + warp * kStages;
  unsigned char* stages = smem_raw + kRowBarBytes + (size_t)warp * kStages * kStageBytes;

  const int K = p.k, V = p.vocab, nc = p.nc, G = p.groups, C = p.slot_cap;
  const int units = (int)p.units;
  const int nwarps = gridDim.x * kRowWarps;
  const int gw = blockIdx.x * kRowWarps + warp;
  const int n_mine = gw < units ? (units - gw + nwarps - 1) / nwarps : 0;
  const unsigned char* logits = static_cast<const unsigned char*>(p.logits);
  const int row_bytes = V * ES;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_barrier_init();
  }
  __syncwarp();
  // the fine-rank kernel may be scheduled from now on: its CTAs take the SM space this
  // grid's CTAs free as they finish, and wait for the whole grid before reading its output
  grid_launch_dependents();
  // this grid may itself start while the previous kernel of the stream finishes (the cache
  // refresh of the previous decode step): wait for it before reading any input
  grid_dependency_wait();

  auto row_of = [&](int u) -> int { return (int)fast_div((uint32_t)u, p.nc_magic, p.nc_shift); };
  auto live = [&](int u) -> bool { return !(p.finished && p.finished[row_of(u)]); };
  struct Geo {
    const unsigned char* rb;  // 16-byte aligned start of the row's first vector
    int lead;                 // bytes of that vector before the row starts
    int j0;                   // first vector of the chunk within the row
    int nvec;                 // vectors in the chunk
  };
  auto geometry = [&](int u) -> Geo {
    Geo g;
    const int row = row_of(u);
    const int c = u - row * nc;
    const unsigned char* rowp = logits + (size_t)row * row_bytes;
    g.lead = (int)(reinterpret_cast<uintptr_t>(rowp) & 15);
    g.rb = rowp - g.lead;
    const int nv = (g.lead + row_bytes + 15) >> 4;
    g.j0 = c * CV;
    g.nvec = max(0, min(CV, nv - g.j0));
    return g;
  };

  // producer state (lane 0)
  int iss_i = 0, n_iss = 0;
  uint64_t policy = 0;
  if (lane == 0) policy = l2_evict_first_policy();
  auto fill = [&](int n_done) {
    while (n_iss - n_done < kStages && iss_i < n_mine) {
      const int u = gw + iss_i * nwarps;
      if (live(u)) {
        const Geo g = geometry(u);
        const int s = n_iss % kStages;
        const uint32_t bar = smem_addr(&bars[s]);
        const uint32_t bytes = (uint32_t)g.nvec * 16u;
        mbar_arrive_expect_tx(bar, bytes);
        if (bytes)
          bulk_load(smem_addr(stages + (size_t)s * kStageBytes), g.rb + (size_t)g.j0 * 16, bytes, bar, policy);
        ++n_iss;
      }
      ++iss_i;
    }
  };
  if (lane == 0) fill(0);

  int n_cons = 0;
  bool aborted = false;
  for (int i = 0; i < n_mine; ++i) {
    const int u = gw + i * nwarps;
    if (!live(u)) continue;
    const Geo g = geometry(u);
    const int s = n_cons % kStages;
    const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (uint32_t)((n_cons / kStages) & 1), p.spin_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      aborted = true;
      break;
    }
    // the chunk into registers; bytes outside the row become -inf
    const uint4* sv = reinterpret_cast<const uint4*>(stages + (size_t)s * kStageBytes);
    uint4 d[VPL];
    // a chunk of CV whole vectors that starts and ends inside the row needs no masking
    const bool interior_chunk = g.nvec == CV && g.j0 * 16 - g.lead >= 0 && (g.j0 + CV) * 16 - g.lead <= row_bytes;
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      const int jl = lane + 32 * r;
      if (interior_chunk) {
        d[r] = sv[jl];
      } else if (jl < g.nvec) {
        d[r] = sv[jl];
        const int base_b = (g.j0 + jl) * 16 - g.lead;  // row byte offset of element 0
        if (base_b < 0 || base_b + 16 > row_bytes) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const int eb = base_b + e * ES;
            if (eb < 0 || eb >= row_bytes) set_neg_inf<DT>(d[r], e);
          }
        }
      } else {
        const uint32_t w = Traits<DT>::kNegInfWord;
        d[r] = make_uint4(w, w, w, w);
      }
    }

    // x = logit + bias of local vector jl's element e (bias only for tokens inside the row)
    auto bias_of = [&](int jl, int e) -> float {
      const int eb = (g.j0 + jl) * 16 - g.lead + e * ES;
      return (eb >= 0 && eb < row_bytes) ? __ldg(p.bias + eb / ES) : 0.0f;
    };
    // with a bias the chunk is converted once to x = logit + bias, kept as floats
    float xb[BIAS ? VPL * VEC : 1];
    if constexpr (BIAS) {
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        float x[VEC];
        unpack<DT>(d[r], x);
        const int jl = lane + 32 * r;
        const int base_b = (g.j0 + jl) * 16 - g.lead;
        const int v0 = base_b / ES;  // token id of element 0 (negative before the row start)
        if (jl < g.nvec) {
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
            for (int e = 0; e < VEC; ++e) x[e] += bias_of(jl, e);
          }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) xb[r * VEC + e] = x[e];
      }
    }

    // first traversal, part 1: per-vector maxima (packed), lane and chunk maxima
    uint32_t vm[VPL];
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      if constexpr (BIAS) {
        float mr = xb[r * VEC];
#pragma unroll
        for (int e = 1; e < VEC; ++e) mr = fmaxf(mr, xb[r * VEC + e]);
        vm[r] = __float_as_uint(mr);
      } else {
        vm[r] = vec_max_bits<DT>(d[r]);
      }
    }
    constexpr int BT = BIAS ? DT_F32 : DT;  // type of the packed maxima
    uint32_t b0 = vm[0], b1 = VPL > 1 ? vm[1] : vm[0];
#pragma unroll
    for (int r = 2; r < VPL; r += 2) {
      b0 = max_bits<BT>(b0, vm[r]);
      if (r + 1 < VPL) b1 = max_bits<BT>(b1, vm[r + 1]);
    }
    const float m0 = bits_max_float<BT>(b0);  // even vectors (group lane when G = 64)
    const float m1 = VPL > 1 ? bits_max_float<BT>(b1) : -INFINITY;  // odd vectors (group lane + 32)
    const float mt = fmaxf(m0, m1);
    // group maxima, the chunk max M and the chunk's R-top-k
    float* rec = reinterpret_cast<float*>(p.rec + (size_t)u * p.rec_stride);
    float M, rt;
    if (G <= 32) {
      float gmv = mt;
      for (int o = 16; o >= G; o >>= 1) gmv = fmaxf(gmv, __shfl_xor_sync(0xffffffffu, gmv, o));
      if (lane < G) rec[4 + lane] = gmv;
      // the remaining levels of the same tree give the chunk max and the least group max,
      // which is the k-th largest of the G group maxima when G = k
      float mx = gmv, mn = gmv;
      for (int o = G >> 1; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      }
      M = mx;
      rt = (G == K) ? mn : warp_kth_of_lanes(gmv, G, K);
    } else {
      M = warp_max(mt);
      rec[4 + lane] = m0;
      rec[4 + 32 + lane] = m1;
      rt = warp_kth_of_64(m0, m1, K);
    }

    // second traversal: survivors x >= rt.  The vectors whose max reaches rt are listed in
    // the warp's shared list (one item per vector, up to 32 items a round, one item per
    // lane) and re-read from the stage, which is still in shared memory.
    int* wlist = reinterpret_cast<int*>(smem_raw + kRowListOff) + warp * 32;
    const unsigned lt_mask = (1u << lane) - 1u;
    uint32_t qm[VPL];
    auto list_items = [&](float thr) -> int {
      const uint32_t t2 = thr_bits<BT>(thr);
      int n = 0;
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        qm[r] = __ballot_sync(0xffffffffu, packed_ge<BT>(vm[r], t2));
        n += __popc(qm[r]);
      }
      return n;
    };
    // fill the list with items [base, base + 32); returns the item count of the round
    auto fill_list = [&](int base, int n) -> int {
      int pre = 0;
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        if ((qm[r] >> lane) & 1u) {
          const int pos = pre + __popc(qm[r] & lt_mask) - base;
          if (pos >= 0 && pos < 32) wlist[pos] = (r << 5) | lane;
        }
        pre += __popc(qm[r]);
      }
      __syncwarp();
      return min(32, n - base);
    };
    // survivor mask of one listed vector (bit e: element e is in the row and >= thr)
    auto item_mask = [&](int jl, const uint4& raw, float thr) -> uint32_t {
      const int base_b = (g.j0 + jl) * 16 - g.lead;
      const bool interior = base_b >= 0 && base_b + 16 <= row_bytes;
      uint32_t mr;
      if constexpr (BIAS) {
        float x[VEC];
        unpack<DT>(raw, x);
        mr = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const int eb = base_b + e * ES;
          const bool in_row = eb >= 0 && eb < row_bytes;
          const float xe = x[e] + (in_row ? __ldg(p.bias + eb / ES) : 0.0f);
          mr |= (in_row && xe >= thr ? 1u : 0u) << e;
        }
      } else {
        mr = vec_ge_mask<DT>(raw, thr);
        if (!interior) {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const int eb = base_b + e * ES;
            if (eb < 0 || eb >= row_bytes) mr &= ~(1u << e);
          }
        }
      }
      return jl < g.nvec ? mr : 0u;
    };
    // survivors, one round of up to 32 listed vectors at a time; masks are computed once
    // per round and written at once unless the chunk overflows its slots, in which case
    // the bound is tightened (k <= 32) and the chunk filtered again
    CandSlot* slots = p.slots + (size_t)u * C;
    auto filter = [&](float thr, int n, bool write) -> int {
      int written = 0;
      for (int base = 0; base < n; base += 32) {
        const int m = fill_list(base, n);
        uint32_t mr = 0;
        uint4 raw = make_uint4(0, 0, 0, 0);
        int jl = 0;
        if (lane < m) {
          const int it = wlist[lane];
          jl = (it & 31) + 32 * (it >> 5);
          raw = sv[jl];
          mr = item_mask(jl, raw, thr);
        }
        __syncwarp();
        const int c = __popc(mr);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        if (write) {
          int pos = written + incl - c;
          const int base_b = (g.j0 + jl) * 16 - g.lead;
          while (mr) {
            const int e = __ffs(mr) - 1;
            mr &= mr - 1;
            if (pos < C) {
              const int eb = base_b + e * ES;
              CandSlot cs;
              float x = vec_elem<DT>(raw, e);
              if constexpr (BIAS) x += __ldg(p.bias + eb / ES);
              cs.x = x;
              cs.v = eb / ES;
              slots[pos] = cs;
            }
            ++pos;
          }
        }
        written += __shfl_sync(0xffffffffu, incl, 31);
      }
      return written;
    };
    int n_items = list_items(rt);
    // common case: everything fits, count and write in one pass (every listed vector
    // holds at least one survivor, so more than C vectors means more than C survivors)
    int total = (n_items <= C) ? filter(rt, n_items, true) : C + 1;
    if (total > C) {
      if (K <= 32) {
        // tighter bound: k-th largest of the 32 per-lane maxima (32 disjoint groups)
        rt = fmaxf(rt, warp_kth_of_lanes(mt, 32, K));
        n_items = list_items(rt);
      }
      total = filter(rt, n_items, false);
      if (total <= C) filter(rt, n_items, true);
    }
    __syncwarp();
    ++n_cons;
    if (lane == 0) fill(n_cons);  // the stage is free again: the next copy lands during the sum

    // first traversal, part 2: sum of exp(x - M) = 2^((x - M) log2 e) with packed fp32x2.
    // For |M| < 64, x log2e - M log2e in one fused multiply-add (the rounding of M log2e
    // shifts every term alike, by at most 2^-18 in the exponent); otherwise the exact
    // difference x - M first (exact for the terms that dominate the sum).
    float ssum = 0.0f;
    if (M != -INFINITY) {
      const float2 L2 = make_float2(kLog2e, kLog2e);
      float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
      if (fabsf(M) < 64.0f) {
        const float2 nml = make_float2(-M * kLog2e, -M * kLog2e);
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
          float x[VEC];
          if constexpr (BIAS) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) x[e] = xb[r * VEC + e];
          } else {
            unpack<DT>(d[r], x);
          }
#pragma unroll
          for (int e = 0; e < VEC; e += 4) {
            const float2 t0 = __ffma2_rn(make_float2(x[e], x[e + 1]), L2, nml);
            const float2 t1 = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), L2, nml);
            acc0 = __fadd2_rn(acc0, make_float2(fast_exp2(t0.x), fast_exp2(t0.y)));
            acc1 = __fadd2_rn(acc1, make_float2(fast_exp2(t1.x), fast_exp2(t1.y)));
          }
        }
      } else {
        const float2 nm = make_float2(-M, -M);
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
          float x[VEC];
          if constexpr (BIAS) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) x[e] = xb[r * VEC + e];
          } else {
            unpack<DT>(d[r], x);
          }
#pragma unroll
          for (int e = 0; e < VEC; e += 4) {
            const float2 t0 = __fmul2_rn(__fadd2_rn(make_float2(x[e], x[e + 1]), nm), L2);
            const float2 t1 = __fmul2_rn(__fadd2_rn(make_float2(x[e + 2], x[e + 3]), nm), L2);
            acc0 = __fadd2_rn(acc0, make_float2(fast_exp2(t0.x), fast_exp2(t0.y)));
            acc1 = __fadd2_rn(acc1, make_float2(fast_exp2(t1.x), fast_exp2(t1.y)));
          }
        }
      }
      const float2 a = __fadd2_rn(acc0, acc1);
      ssum = a.x + a.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (lane == 0) {
      reinterpret_cast<int*>(rec)[0] = total;
      rec[1] = M;
      rec[2] = ssum;
    }
  }

  if (aborted && lane == 0) {
    // a wait ran out: record it, then let every copy this warp issued land before exit
    atomicOr(p.status, kDevTimeout);
    for (int n = n_cons; n < n_iss; ++n)
      mbar_wait_bounded(smem_addr(&bars[n % kStages]), (uint32_t)((n / kStages) & 1), kDrainLimitNs);
  }
  __syncwarp();
}

template <int DT, bool BIAS, int VPL>
cudaError_t launch_t(const StepParams& p, int grid, cudaStream_t stream) {
  const size_t smem = beam_rows_smem_bytes(VPL);
  PdlLaunch l(dim3((unsigned)grid), dim3(kRowThreads), smem, stream);
  return cudaLaunchKernelEx(&l.cfg, beam_rows_kernel<DT, BIAS, VPL>, p);
}

template <int DT, bool BIAS, int VPL>
cudaError_t config_t(int* occ) {
  auto fn = beam_rows_kernel<DT, BIAS, VPL>;
  const size_t smem = beam_rows_smem_bytes(VPL);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kRowThreads, smem);
}

template <int DT, bool BIAS>
cudaError_t dispatch_vpl(bool launch, const StepParams* p, int vpl, int grid, cudaStream_t stream, int* occ) {
  switch (vpl) {
    case 4: return launch ? launch_t<DT, BIAS, 4>(*p, grid, stream) : config_t<DT, BIAS, 4>(occ);
    case 8: return launch ? launch_t<DT, BIAS, 8>(*p, grid, stream) : config_t<DT, BIAS, 8>(occ);
    case 16: return launch ? launch_t<DT, BIAS, 16>(*p, grid, stream) : config_t<DT, BIAS, 16>(occ);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch(bool launch, const StepParams* p, int dtype, bool bias, int vpl, int grid, cudaStream_t stream,
                     int* occ) {
  switch (dtype) {
    case DT_F32:
      return bias ? dispatch_vpl<DT_F32, true>(launch, p, vpl, grid, stream, occ)
                  : dispatch_vpl<DT_F32, false>(launch, p, vpl, grid, stream, occ);
    case DT_F16:
      return bias ? dispatch_vpl<DT_F16, true>(launch, p, vpl, grid, stream, occ)
                  : dispatch_vpl<DT_F16, false>(launch, p, vpl, grid, stream, occ);
    case DT_BF16:
      return bias ? dispatch_vpl<DT_BF16, true>(launch, p, vpl, grid, stream, occ)
                  : dispatch_vpl<DT_BF16, false>(launch, p, vpl, grid, stream, occ);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t beam_rows_smem_bytes(int vpl) {
  return kRowBarBytes + (size_t)kRowWarps * stages_for(vpl) * 32 * vpl * 16;
}

cudaError_t beam_rows_config(int dtype, bool bias, int vpl, int* occupancy) {
  return dispatch(false, nullptr, dtype, bias, vpl, 0, nullptr, occupancy);
}

cudaError_t launch_beam_rows(const StepParams& p, int dtype, int vpl, int grid, cudaStream_t stream) {
  return dispatch(true, &p, dtype, p.bias != nullptr, vpl, grid, stream, nullptr);
}

}  // namespace lsb
