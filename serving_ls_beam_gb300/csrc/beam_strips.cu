// Beam-step kernel K1s: the first and second traversal of every beam's logits, each row
// (or each of a few interleaved strips of it) streamed start to end by one warp.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), hierarchical decoding
// section.  First traversal: split a beam's logits into groups, take each group's max; the
// k-th largest of those maxima (their min when there are exactly k groups) is the R-top-k
// bound, never above the true k-th largest; log_sum_exp in the same pass.  Second
// traversal: keep the logits at or above R-top-k as candidates.
//
// GB300 design:
//  * Work unit = one strip of one beam's row: the row is cut into stages of 32 x VPL
//    16-byte vectors and strip w of W takes stages w, w + W, ...  A warp owns a unit from
//    its first stage to its last; lane 0 keeps a ring of `stages` shared-memory buffers full
//    with 1-D bulk (TMA) copies (L2 evict-first) completed on per-stage mbarriers, and the
//    ring runs on into the warp's next unit.  No CTA barrier and no global atomic: the
//    warps of a CTA are independent.
//  * Both traversals run on the stage in registers.  Groups are the lanes modulo G (G = the
//    power of two >= k): lane l's running max covers every element it has read of the strip.
//    After the maxima of a stage are in, the bound R = k-th largest of the G running group
//    maxima is a lower bound of the row's k-th largest x that only rises along the strip,
//    so a candidate dropped against the R of its stage is below every later bound too.  The
//    second traversal keeps the elements x >= R of the stage in a per-warp list (a few per
//    stage at the start of a row, almost none later); at the end of the strip the list is
//    filtered once more against the strip's final R and written as the unit's slots.
//  * log_sum_exp: a running (max, sum of exp(x - max)) per lane, rescaled when the lane's
//    max rises; the difference x - max is formed exactly (for 16-bit logits by the mixed
//    f16/bf16 -> f32 subtraction), then scaled by log2 e for ex2.
//  * Output per unit: K1's chunk record (count, max, sum, group maxima) and slots, so the
//    fine rank K2 (beam_select.cu) runs unchanged with W "chunks" per row.
#include "ls_device.cuh"
#include "ls_dtype.cuh"
#include "ls_internal.h"
#include "ls_strip.cuh"

namespace lsb {
namespace {

constexpr long long kDrainLimitNs = 2000000000LL;  // 2 s for copies already in flight

static_assert(kStWarps * kStMaxStages * 8 <= kStListOff, "mbarriers overlap the lists");
static_assert(kStBarBytes % 16 == 0, "stage buffers must be 16-byte aligned for bulk copies");

template <int DT, bool BIAS, int VPL>
__global__ void __launch_bounds__(kStThreads, 3) beam_strips_kernel(const StepParams p) {
  constexpr int VEC = Traits<DT>::kVec;
  constexpr int ES = Traits<DT>::kBytes;
  constexpr int CV = 32 * VPL;  // vectors per stage
  constexpr uint32_t kStageBytes = CV * 16;
  constexpr bool kPacked = (DT != DT_F32) && !BIAS;  // pass 1 on packed 16-bit pairs
  constexpr int EL = VPL * VEC;                      // elements per lane per stage
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int S = p.stages;
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(smem_raw) + warp * kStMaxStages;
  float2* list = reinterpret_cast<float2*>(smem_raw + kStListOff) + warp * kStListCap;
  unsigned char* stages = smem_raw + kStBarBytes + (size_t)warp * S * kStageBytes;

  const int K = p.k, V = p.vocab, W = p.nc, G = p.groups, C = p.slot_cap;
  const int units = (int)p.units;
  const int nwarps = gridDim.x * kStWarps;
  const int gw = blockIdx.x * kStWarps + warp;
  const unsigned char* logits = static_cast<const unsigned char*>(p.logits);
  const int row_bytes = V * ES;
  const float lo_fin = lowest_finite<DT>();

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_barrier_init();
  }
  __syncwarp();
  // the fine-rank kernel may be scheduled from now on (it waits for this whole grid)
  grid_launch_dependents();
  // inputs may come from the previous kernel of the stream
  grid_dependency_wait();

  // A unit's geometry: its row's 16-byte aligned vectors and the stages of its strip.
  struct Unit {
    int u;                    // unit index (>= units: none)
    const unsigned char* rb;  // 16-byte aligned start of the row's first vector
    int lead;                 // bytes of that vector before the row starts
    int nv;                   // vectors covering the row
    int ns;                   // stages of the row; the strip's are part, part + W, ...
    int part;
  };
  // the warp's next live unit at or after u (every strip has a stage: W <= stages of a row)
  auto unit_from = [&](int u) -> Unit {
    Unit t;
    for (; u < units; u += nwarps) {
      const int row = (int)fast_div((uint32_t)u, p.nc_magic, p.nc_shift);
      if (p.finished && p.finished[row]) continue;
      const unsigned char* rowp = logits + (size_t)row * row_bytes;
      t.lead = (int)(reinterpret_cast<uintptr_t>(rowp) & 15);
      t.rb = rowp - t.lead;
      t.nv = (t.lead + row_bytes + 15) >> 4;
      t.ns = (t.nv + CV - 1) / CV;
      t.part = u - row * W;
      break;
    }
    t.u = u;
    return t;
  };

  // producer (lane 0): the next stage to copy and the number of copies issued
  Unit pu;
  int pq = 0, n_iss = 0;
  uint64_t policy = 0;
  if (lane == 0) {
    policy = l2_evict_first_policy();
    pu = unit_from(gw);
    pq = pu.part;
  }
  auto issue_one = [&]() {
    if (pu.u >= units) return;
    const int j0 = pq * CV;
    const uint32_t bytes = (uint32_t)min(CV, pu.nv - j0) * 16u;
    const int s = n_iss % S;
    const uint32_t bar = smem_addr(&bars[s]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(smem_addr(stages + (size_t)s * kStageBytes), pu.rb + (size_t)j0 * 16, bytes, bar, policy);
    ++n_iss;
    pq += W;
    if (pq >= pu.ns) {
      pu = unit_from(pu.u + nwarps);
      pq = pu.part;
    }
  };
  if (lane == 0)
    for (int s = 0; s < S; ++s) issue_one();

  int n_cons = 0;
  bool aborted = false;
  for (Unit cu = unit_from(gw); cu.u < units && !aborted; cu = unit_from(cu.u + nwarps)) {
    // running state of the unit
    float ml = -INFINITY, sl = 0.0f;  // lane's running max and sum of exp(x - ml)
    float R = -INFINITY, gm = -INFINITY;
    float Rfl = -INFINITY;  // a tighter bound taken when a stage has many candidates
    int cnt = 0;            // entries in the warp's list
    bool ovf = false;       // the list could not hold the candidates
    // keep the list's entries x >= t, in order; returns their count
    auto drop_below = [&](int n_in, float t) -> int {
      int out = 0;
      for (int b0 = 0; b0 < n_in; b0 += 32) {
        const int i = b0 + lane;
        const float2 en = i < n_in ? list[i] : make_float2(-INFINITY, 0.0f);
        const bool keep = i < n_in && en.x >= t;
        const unsigned bm = __ballot_sync(0xffffffffu, keep);
        __syncwarp();
        if (keep) list[out + __popc(bm & ((1u << lane) - 1u))] = en;
        out += __popc(bm);
        __syncwarp();
      }
      return out;
    };
    for (int q = cu.part; q < cu.ns; q += W) {
      const int s = n_cons % S;
      const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), (uint32_t)((n_cons / S) & 1), p.spin_limit_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        aborted = true;
        break;
      }
      const int j0 = q * CV;
      const int nvec = min(CV, cu.nv - j0);
      const uint4* sv = reinterpret_cast<const uint4*>(stages + (size_t)s * kStageBytes);
      uint4 d[VPL];
      const bool interior = nvec == CV && j0 * 16 - cu.lead >= 0 && (j0 + CV) * 16 - cu.lead <= row_bytes;
      if (interior) {
#pragma unroll
        for (int r = 0; r < VPL; ++r) d[r] = sv[lane + 32 * r];
      } else {
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
          const int jl = lane + 32 * r;
          if (jl < nvec) {
            d[r] = sv[jl];
            const int base_b = (j0 + jl) * 16 - cu.lead;  // row byte offset of element 0
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
      }
      // the stage is in registers: hand it back to the producer
      __syncwarp();
      ++n_cons;
      if (lane == 0) issue_one();

      // x = logit + bias as floats (bias and f32 variants)
      float xf[kPacked ? 1 : EL];
      if constexpr (!kPacked) {
#pragma unroll
        for (int r = 0; r < VPL; ++r) {
          float x[VEC];
          unpack<DT>(d[r], x);
          if constexpr (BIAS) {
            const int base_b = (j0 + lane + 32 * r) * 16 - cu.lead;
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
      }

      // first traversal: the lane's stage max, the running maxima and R
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
      const float mn = fmaxf(ml, lm);
      R = fmaxf(strip_bound(mn, G, K, gm), Rfl);
      float thr = fmaxf(R, lo_fin);

      // second traversal: the stage's candidates x >= R into the warp's list
      if (__any_sync(0xffffffffu, lm >= thr)) {
        // bit r * VEC + e: element e of vector r is >= t
        auto stage_mask = [&](float t) -> uint64_t {
          uint64_t mk = 0;
          if (lm >= t) {
#pragma unroll
            for (int r = 0; r < VPL; ++r) {
              uint32_t m;
              if constexpr (kPacked) {
                m = hvec_ge_mask<DT>(d[r], t);
              } else {
                m = 0;
#pragma unroll
                for (int e = 0; e < VEC; ++e) m |= (xf[r * VEC + e] >= t ? 1u : 0u) << e;
              }
              mk |= (uint64_t)m << (r * VEC);
            }
          }
          return mk;
        };
        uint64_t mk = stage_mask(thr);
        int n = __reduce_add_sync(0xffffffffu, __popcll(mk));
        if (n > kStTighten) {
          // many candidates (a wide spread of group maxima, e.g. heavy tails): raise the
          // bound to the k-th largest of the 32 lanes' running maxima (32 disjoint groups)
          Rfl = fmaxf(Rfl, kth_of_lanes(mn, 32, K));
          R = fmaxf(R, Rfl);
          thr = fmaxf(R, lo_fin);
          mk = stage_mask(thr);
          n = __reduce_add_sync(0xffffffffu, __popcll(mk));
        }
        if (!ovf && cnt + n > kStListCap) {
          // drop the entries below the current bound (it only rises along the strip)
          cnt = drop_below(cnt, thr);
          if (cnt + n > kStListCap) {
            // still more than the list holds: the k-th largest of the list and the stage's
            // candidates together is itself a lower bound of the row's k-th largest (they are
            // elements of the row).  Raise the bound to it -- the largest value t of the
            // compared type with at least k of them >= t, by bisection on its order key.
            auto count_ge = [&](float t) -> int {
              int nge = __reduce_add_sync(0xffffffffu, __popcll(stage_mask(t)));
              for (int b0 = 0; b0 < cnt; b0 += 32) {
                const int i = b0 + lane;
                nge += __popc(__ballot_sync(0xffffffffu, i < cnt && list[i].x >= t));
              }
              return nge;
            };
            float hv = lm;
            for (int i = lane; i < cnt; i += 32) hv = fmaxf(hv, list[i].x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, o));
            using OK = OrderKey<DT, kPacked>;
            float kb = hv;
            if (count_ge(hv) < K) {
              uint32_t lo = OK::of(thr), hi = OK::of(hv);  // count_ge(lo) >= k > count_ge(hi)
              while (hi - lo > 1u) {
                const uint32_t mid = lo + ((hi - lo) >> 1);
                if (count_ge(OK::val(mid)) >= K)
                  lo = mid;
                else
                  hi = mid;
              }
              kb = OK::val(lo);
            }
            Rfl = fmaxf(Rfl, kb);
            R = fmaxf(R, Rfl);
            thr = fmaxf(R, lo_fin);
            cnt = drop_below(cnt, thr);
            mk = stage_mask(thr);
            n = __reduce_add_sync(0xffffffffu, __popcll(mk));
          }
          if (cnt + n > kStListCap) ovf = true;  // ties at the bound beyond the list
        }
        const int c = __popcll(mk);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        if (!ovf) {
          int pos = cnt + incl - c;
#pragma unroll
          for (int r = 0; r < VPL; ++r) {
            uint32_t m = (uint32_t)(mk >> (r * VEC)) & ((1u << VEC) - 1u);
            while (m) {
              const int e = __ffs(m) - 1;
              m &= m - 1;
              const int eb = (j0 + lane + 32 * r) * 16 - cu.lead + e * ES;
              float x;
              if constexpr (kPacked) {
                x = vec_elem_f<DT>(d[r], e);
              } else {
                float t = xf[r * VEC];
#pragma unroll
                for (int q2 = 1; q2 < VEC; ++q2) t = q2 == e ? xf[r * VEC + q2] : t;
                x = t;
              }
              list[pos++] = make_float2(x, __int_as_float(eb / ES));
            }
          }
          cnt += n;
        }
        __syncwarp();
      }

      // first traversal, log_sum_exp: sum of exp(x - mn) = 2^((x - mn) log2 e).  For
      // |mn| < 64, x log2e - mn log2e in one fused multiply-add (the rounding of mn log2e
      // scales every term of this lane and stage alike, by at most 2^-17 relative);
      // otherwise the exact difference x - mn first.
      if (mn != ml) {
        sl = (ml == -INFINITY) ? 0.0f : sl * fast_exp2((ml - mn) * kLog2e);
        ml = mn;
      }
      if (ml != -INFINITY) {
        const float2 L2 = make_float2(kLog2e, kLog2e);
        float2 a0 = make_float2(0.0f, 0.0f), a1 = make_float2(0.0f, 0.0f);
        const bool fused = fabsf(ml) < 64.0f;
        const float2 nml = fused ? make_float2(-ml * kLog2e, -ml * kLog2e) : make_float2(-ml, -ml);
        auto term2 = [&](float2 x) -> float2 {
          const float2 t = fused ? __ffma2_rn(x, L2, nml) : __fmul2_rn(__fadd2_rn(x, nml), L2);
          return make_float2(fast_exp2(t.x), fast_exp2(t.y));
        };
        if constexpr (kPacked) {
#pragma unroll
          for (int r = 0; r < VPL; ++r) {
            const uint32_t w[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
              float2 f0, f1;
              if constexpr (DT == DT_F16) {
                f0 = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
                f1 = __half22float2(*reinterpret_cast<const __half2*>(&w[i + 1]));
              } else {
                f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i + 1]));
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
    }
    if (aborted) break;

    // end of the unit: merge the lanes' (max, sum), filter the list by the final R, write
    // the record and the slots
    float M = ml;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float sm = (ml == -INFINITY) ? 0.0f : sl * fast_exp2((ml - M) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    float thr = fmaxf(R, lo_fin);
    auto count_above = [&](float t) -> int {
      int n = 0;
      for (int b0 = 0; b0 < cnt; b0 += 32) {
        const int i = b0 + lane;
        n += __popc(__ballot_sync(0xffffffffu, i < cnt && list[i].x >= t));
      }
      return n;
    };
    if (!ovf && count_above(thr) > C) {
      // more than the slots hold: the tighter bound of the 32 lanes' maxima, then, if still
      // too many, the k-th largest of the list itself (bisection as above)
      R = fmaxf(R, kth_of_lanes(ml, 32, K));
      thr = fmaxf(R, lo_fin);
      if (count_above(thr) > C) {
        using OK = OrderKey<DT, kPacked>;
        float hv = -INFINITY;
        for (int i = lane; i < cnt; i += 32) hv = fmaxf(hv, list[i].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) hv = fmaxf(hv, __shfl_xor_sync(0xffffffffu, hv, o));
        float kb = hv;
        if (count_above(hv) < K) {
          uint32_t lo = OK::of(thr), hi = OK::of(hv);
          while (hi - lo > 1u) {
            const uint32_t mid = lo + ((hi - lo) >> 1);
            if (count_above(OK::val(mid)) >= K)
              lo = mid;
            else
              hi = mid;
          }
          kb = OK::val(lo);
        }
        R = fmaxf(R, kb);
        thr = fmaxf(R, lo_fin);
      }
    }
    CandSlot* slots = p.slots + (size_t)cu.u * C;
    int total = 0;
    for (int b0 = 0; b0 < cnt; b0 += 32) {
      const int i = b0 + lane;
      const float2 en = i < cnt ? list[i] : make_float2(-INFINITY, 0.0f);
      const bool keep = i < cnt && en.x >= thr;
      const unsigned bm = __ballot_sync(0xffffffffu, keep);
      const int pos = total + __popc(bm & ((1u << lane) - 1u));
      if (keep && pos < C) {
        CandSlot cs;
        cs.x = en.x;
        cs.v = __float_as_int(en.y);
        slots[pos] = cs;
      }
      total += __popc(bm);
    }
    if (ovf) total = C + 1;  // the fine rank takes its exact path for this batch
    float* rec = reinterpret_cast<float*>(p.rec + (size_t)cu.u * p.rec_stride);
    if (lane < G) rec[4 + lane] = gm;
    if (lane == 0) {
      reinterpret_cast<int*>(rec)[0] = total;
      rec[1] = M;
      rec[2] = sm;
    }
    __syncwarp();
  }

  if (aborted && lane == 0) {
    // a wait ran out: record it, then let every copy this warp issued land before exit
    atomicOr(p.status, kDevTimeout);
    for (int n = n_cons; n < n_iss; ++n)
      mbar_wait_bounded(smem_addr(&bars[n % S]), (uint32_t)((n / S) & 1), kDrainLimitNs);
  }
  __syncwarp();
}

template <int DT, bool BIAS, int VPL>
cudaError_t launch_t(const StepParams& p, int grid, cudaStream_t stream) {
  const size_t smem = beam_strips_smem_bytes(VPL, p.stages);
  PdlLaunch l(dim3((unsigned)grid), dim3(kStThreads), smem, stream);
  return cudaLaunchKernelEx(&l.cfg, beam_strips_kernel<DT, BIAS, VPL>, p);
}

template <int DT, bool BIAS, int VPL>
cudaError_t config_t(int stages, int* occ) {
  auto fn = beam_strips_kernel<DT, BIAS, VPL>;
  const size_t smem = beam_strips_smem_bytes(VPL, stages);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kStThreads, smem);
}

template <int DT, bool BIAS>
cudaError_t dispatch_vpl(bool launch, const StepParams* p, int vpl, int stages, int grid, cudaStream_t stream,
                         int* occ) {
  switch (vpl) {
    case 4: return launch ? launch_t<DT, BIAS, 4>(*p, grid, stream) : config_t<DT, BIAS, 4>(stages, occ);
    case 8: return launch ? launch_t<DT, BIAS, 8>(*p, grid, stream) : config_t<DT, BIAS, 8>(stages, occ);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t dispatch(bool launch, const StepParams* p, int dtype, bool bias, int vpl, int stages, int grid,
                     cudaStream_t stream, int* occ) {
  switch (dtype) {
    case DT_F32:
      return bias ? dispatch_vpl<DT_F32, true>(launch, p, vpl, stages, grid, stream, occ)
                  : dispatch_vpl<DT_F32, false>(launch, p, vpl, stages, grid, stream, occ);
    case DT_F16:
      return bias ? dispatch_vpl<DT_F16, true>(launch, p, vpl, stages, grid, stream, occ)
                  : dispatch_vpl<DT_F16, false>(launch, p, vpl, stages, grid, stream, occ);
    case DT_BF16:
      return bias ? dispatch_vpl<DT_BF16, true>(launch, p, vpl, stages, grid, stream, occ)
                  : dispatch_vpl<DT_BF16, false>(launch, p, vpl, stages, grid, stream, occ);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t beam_strips_smem_bytes(int vpl, int stages) {
  return kStBarBytes + (size_t)kStWarps * stages * 32 * vpl * 16;
}

cudaError_t beam_strips_config(int dtype, bool bias, int vpl, int stages, int* occupancy) {
  return dispatch(false, nullptr, dtype, bias, vpl, stages, 0, nullptr, occupancy);
}

cudaError_t launch_beam_strips(const StepParams& p, int dtype, int vpl, int grid, cudaStream_t stream) {
  return dispatch(true, &p, dtype, p.bias != nullptr, vpl, p.stages, grid, stream, nullptr);
}

}  // namespace lsb
