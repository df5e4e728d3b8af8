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

constexpr int kStages = 2;
constexpr long long kDrainLimitNs = 2000000000LL;  // 2 s for copies already in flight

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
    rank += (w > v) || (w == v && q < lane);
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
    ra += (wa > a) || (wa == a && q < lane);
    ra += (wb > a);
    rb += (wa >= b);
    rb += (wb > b) || (wb == b && q < lane);
  }
  const bool ha = ra == k - 1, hb = rb == k - 1;
  const unsigned hit = __ballot_sync(0xffffffffu, ha || hb);
  const float mine = ha ? a : b;
  return __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1);
}

// Max of the VEC values of a 16-byte vector (values before any bias).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& d) {
  if constexpr (DT == DT_F32) {
    return fmaxf(fmaxf(__uint_as_float(d.x), __uint_as_float(d.y)), fmaxf(__uint_as_float(d.z), __uint_as_float(d.w)));
  } else if constexpr (DT == DT_F16) {
    const __half2* h = reinterpret_cast<const __half2*>(&d);
    const __half2 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(m), __high2float(m));
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&d);
    const __nv_bfloat162 m = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(m), __high2float(m));
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
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t g;
      if constexpr (DT == DT_F16) {
        const __half2 t = __float2half2_rn(thr);
        g = __hge2_mask(*reinterpret_cast<const __half2*>(&w[i]), t);
      } else {
        const __nv_bfloat162 t = __float2bfloat162_rn(thr);
        g = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[i]), t);
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
__global__ void __launch_bounds__(kRowThreads, 3) beam_rows_kernel(const StepParams p) {
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
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      const int jl = lane + 32 * r;
      if (jl < g.nvec) {
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
    __syncwarp();
    ++n_cons;
    if (lane == 0) fill(n_cons);  // the stage just read is free again

    // x = logit + bias of vector r (bias only: the values without bias are d[r] itself)
    auto add_bias = [&](int r, float (&x)[VEC]) {
      if constexpr (BIAS) {
        const int jl = lane + 32 * r;
        if (jl < g.nvec) {
          const int base_b = (g.j0 + jl) * 16 - g.lead;
          const int v0 = base_b / ES;  // token id of element 0 (negative before the row start)
          const bool interior = base_b >= 0 && base_b + 16 <= row_bytes;
          if (interior && ((reinterpret_cast<uintptr_t>(p.bias + v0) & 15) == 0)) {
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
              const int v = v0 + e;
              if (v >= 0 && v < V) x[e] += __ldg(p.bias + v);
            }
          }
        }
      }
    };
    // with a bias the chunk is converted once to x = logit + bias, kept as floats
    float xb[BIAS ? VPL * VEC : 1];
    if constexpr (BIAS) {
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        float x[VEC];
        unpack<DT>(d[r], x);
        add_bias(r, x);
#pragma unroll
        for (int e = 0; e < VEC; ++e) xb[r * VEC + e] = x[e];
      }
    }

    // first traversal, part 1: per-vector maxima
    float vmax[VPL];
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      if constexpr (BIAS) {
        float mr = xb[r * VEC];
#pragma unroll
        for (int e = 1; e < VEC; ++e) mr = fmaxf(mr, xb[r * VEC + e]);
        vmax[r] = mr;
      } else {
        vmax[r] = vec_max<DT>(d[r]);
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY;  // even / odd vectors (the two groups of a lane when G = 64)
#pragma unroll
    for (int r = 0; r < VPL; r += 2) {
      m0 = fmaxf(m0, vmax[r]);
      if (r + 1 < VPL) m1 = fmaxf(m1, vmax[r + 1]);
    }
    const float mt = fmaxf(m0, m1);
    const float M = warp_max(mt);
    // first traversal, part 2: sum of exp(x - M) = 2^((x - M) log2 e) with packed fp32x2.
    // For |M| < 64, x log2e - M log2e in one fused multiply-add (the rounding of M log2e
    // shifts every term alike, by at most 2^-18 in the exponent); otherwise the exact
    // difference x - M first (exact for the terms that dominate the sum).
    float ssum = 0.0f;
    if (M != -INFINITY) {
      const float2 L2 = make_float2(kLog2e, kLog2e);
      float2 acc = make_float2(0.0f, 0.0f);
      const bool fused = fabsf(M) < 64.0f;
      const float2 nml = make_float2(-M * kLog2e, -M * kLog2e);
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
        for (int e = 0; e < VEC; e += 2) {
          const float2 xv = make_float2(x[e], x[e + 1]);
          const float2 t = fused ? __ffma2_rn(xv, L2, nml) : __fmul2_rn(__fadd2_rn(xv, nm), L2);
          acc = __fadd2_rn(acc, make_float2(fast_exp2(t.x), fast_exp2(t.y)));
        }
      }
      ssum = acc.x + acc.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    // group maxima and the chunk's R-top-k
    float* rec = reinterpret_cast<float*>(p.rec + (size_t)u * p.rec_stride);
    float rt;
    if (G <= 32) {
      float gmv = mt;
      for (int o = 16; o >= G; o >>= 1) gmv = fmaxf(gmv, __shfl_xor_sync(0xffffffffu, gmv, o));
      if (lane < G) rec[4 + lane] = gmv;
      rt = warp_kth_of_lanes(gmv, G, K);
    } else {
      rec[4 + lane] = m0;
      rec[4 + 32 + lane] = m1;
      rt = warp_kth_of_64(m0, m1, K);
    }
    // second traversal: survivors x >= rt.  Only vectors whose max reaches rt are opened;
    // their survivors are kept as bit masks (bit e of mask r = element e of vector r).
    uint32_t mask[VPL];
    auto build = [&](float thr) -> int {
      int c = 0;
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        mask[r] = 0;
        if (__any_sync(0xffffffffu, vmax[r] >= thr) && vmax[r] >= thr) {
          uint32_t mr;
          if constexpr (BIAS) {
            mr = 0;
#pragma unroll
            for (int e = 0; e < VEC; ++e) mr |= (xb[r * VEC + e] >= thr ? 1u : 0u) << e;
          } else {
            mr = vec_ge_mask<DT>(d[r], thr);
          }
          if (thr == -INFINITY) {  // every element passes: drop the ones outside the row
            const int base_b = (g.j0 + lane + 32 * r) * 16 - g.lead;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
              const int eb = base_b + e * ES;
              if (eb < 0 || eb >= row_bytes || lane + 32 * r >= g.nvec) mr &= ~(1u << e);
            }
          }
          mask[r] = mr;
          c += __popc(mr);
        }
      }
      return c;
    };
    int cnt = build(rt);
    int total = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
    if (total > C && K <= 32) {
      // tighter bound: k-th largest of the 32 per-lane maxima (32 disjoint groups)
      rt = fmaxf(rt, warp_kth_of_lanes(mt, 32, K));
      cnt = build(rt);
      total = (int)__reduce_add_sync(0xffffffffu, (unsigned)cnt);
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (cnt) {
      int pos = incl - cnt;
      CandSlot* slots = p.slots + (size_t)u * C;
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        uint32_t mr = mask[r];
        const int base_e = ((g.j0 + lane + 32 * r) * 16 - g.lead) / ES;  // token id of element 0
        while (mr) {
          const int e = __ffs(mr) - 1;
          mr &= mr - 1;
          if (pos < C) {
            CandSlot cs;
            if constexpr (BIAS) {
              float x = xb[r * VEC];
#pragma unroll
              for (int q = 1; q < VEC; ++q)
                if (q == e) x = xb[r * VEC + q];
              cs.x = x;
            } else {
              cs.x = vec_elem<DT>(d[r], e);
            }
            cs.v = base_e + e;
            slots[pos] = cs;
          }
          ++pos;
        }
      }
    }
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
  beam_rows_kernel<DT, BIAS, VPL><<<grid, kRowThreads, smem, stream>>>(p);
  return cudaGetLastError();
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

size_t beam_rows_smem_bytes(int vpl) { return kRowBarBytes + (size_t)kRowWarps * kStages * 32 * vpl * 16; }

cudaError_t beam_rows_config(int dtype, bool bias, int vpl, int* occupancy) {
  return dispatch(false, nullptr, dtype, bias, vpl, 0, nullptr, occupancy);
}

cudaError_t launch_beam_rows(const StepParams& p, int dtype, int vpl, int grid, cudaStream_t stream) {
  return dispatch(true, &p, dtype, p.bias != nullptr, vpl, grid, stream, nullptr);
}

}  // namespace lsb
