// Device helpers of the strip kernels (beam_strips.cu, beam_fused.cu): packed 16-bit
// maxima and comparisons, element extraction, and the R-top-k bound from the lanes'
// running maxima (groups = lanes modulo G).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ls_device.cuh"
#include "ls_dtype.cuh"

namespace lsb {

// Lowest finite value of the element type: a threshold of -inf is raised to it so that
// masked (-inf) elements never count as candidates.
template <int DT>
__device__ __forceinline__ float lowest_finite() {
  if constexpr (DT == DT_F16) return -65504.0f;
  if constexpr (DT == DT_BF16) return -3.3895313892515355e38f;  // 0xff7f: rounds to itself in bf16
  return -3.4028234663852886e38f;
}

// Packed max of two 16-bit pairs (bit patterns).
template <int DT>
__device__ __forceinline__ uint32_t hmax2_bits(uint32_t a, uint32_t b) {
  if constexpr (DT == DT_F16) {
    const __half2 m = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  } else {
    const __nv_bfloat162 m =
        __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&m);
  }
}
template <int DT>
__device__ __forceinline__ float hpair_max(uint32_t a) {
  if constexpr (DT == DT_F16) {
    const __half2 h = *reinterpret_cast<const __half2*>(&a);
    return fmaxf(__low2float(h), __high2float(h));
  } else {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&a);
    return fmaxf(__low2float(h), __high2float(h));
  }
}
// Bits 2i, 2i+1: elements 2i, 2i+1 of the vector are >= t (t an element value of the type,
// so the packed comparison is exact).
template <int DT>
__device__ __forceinline__ uint32_t hvec_ge_mask(const uint4& d, float t) {
  uint32_t tb;
  if constexpr (DT == DT_F16) {
    const __half2 h = __float2half2_rn(t);
    tb = *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __float2bfloat162_rn(t);
    tb = *reinterpret_cast<const uint32_t*>(&h);
  }
  const uint32_t w[4] = {d.x, d.y, d.z, d.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t g;
    if constexpr (DT == DT_F16)
      g = __hge2_mask(*reinterpret_cast<const __half2*>(&w[i]), *reinterpret_cast<const __half2*>(&tb));
    else
      g = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[i]), *reinterpret_cast<const __nv_bfloat162*>(&tb));
    m |= ((g & 1u) | ((g >> 15) & 2u)) << (2 * i);
  }
  return m;
}

// The packed threshold t, t an element value of the type (so packed comparisons are exact).
template <int DT>
__device__ __forceinline__ uint32_t hpack_thr(float t) {
  if constexpr (DT == DT_F16) {
    const __half2 h = __float2half2_rn(t);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __float2bfloat162_rn(t);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}
// Either element of the 16-bit pair w is >= the packed threshold tb.
template <int DT>
__device__ __forceinline__ bool hpair_any_ge(uint32_t w, uint32_t tb) {
  if constexpr (DT == DT_F16)
    return __hge2_mask(*reinterpret_cast<const __half2*>(&w), *reinterpret_cast<const __half2*>(&tb)) != 0u;
  else
    return __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w), *reinterpret_cast<const __nv_bfloat162*>(&tb)) != 0u;
}

// Element e (runtime index) of a 16-byte vector as float, without dynamic register indexing.
template <int DT>
__device__ __forceinline__ float vec_elem_f(const uint4& d, int e) {
  if constexpr (DT == DT_F32) {
    const uint32_t w = e == 0 ? d.x : e == 1 ? d.y : e == 2 ? d.z : d.w;
    return __uint_as_float(w);
  } else {
    const int i = e >> 1;
    const uint32_t w = i == 0 ? d.x : i == 1 ? d.y : i == 2 ? d.z : d.w;
    const unsigned short h = (unsigned short)((e & 1) ? (w >> 16) : (w & 0xffffu));
    if constexpr (DT == DT_F16)
      return __half2float(__ushort_as_half(h));
    else
      return __bfloat162float(__ushort_as_bfloat16(h));
  }
}

// k-th largest (1-based) of the values held by lanes [0, n), n <= 32; all lanes get it.
__device__ __forceinline__ float kth_of_lanes(float v, int n, int k) {
  const int lane = threadIdx.x & 31;
  int rank = 0;
  for (int q = 0; q < n; ++q) {
    const float w = __shfl_sync(0xffffffffu, v, q);
    rank += (w > v) | ((w == v) & (q < lane));
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < n && rank == k - 1);
  return __shfl_sync(0xffffffffu, v, __ffs(hit) - 1);
}

// k-th largest (1-based, k <= 32) of the 32 lanes' values by k rounds of a warp max, each
// taking one lane's value out; all lanes get it.  Cheaper than kth_of_lanes for small k.
__device__ __forceinline__ float kth_by_rounds(float v, int k) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int r = 0; r < k; ++r) {
    m = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const unsigned who = __ballot_sync(0xffffffffu, v == m);
    if (lane == __ffs(who) - 1) v = -INFINITY;
  }
  return m;
}

// Max over the lanes congruent modulo G (offsets 16 .. G), then min over G consecutive
// lanes (offsets G/2 .. 1): with G known at compile time only the needed shuffles run.
template <int G>
__device__ __forceinline__ float lanes_group_max(float v) {
#pragma unroll
  for (int o = 16; o >= G; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int G>
__device__ __forceinline__ float lanes_group_min(float v) {
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int G>
__device__ __forceinline__ float strip_bound_g(float ml, int K, float& gm) {
  const float g = lanes_group_max<G>(ml);
  gm = g;
  return G == 1 ? g : (K == G ? lanes_group_min<G>(g) : kth_of_lanes(g, G, K));
}

// R from the lanes' running maxima: group g = lanes l with l mod G == g; R = k-th largest
// of the G group maxima (their min when G == k).  Lanes g < G return their group max in gm.
__device__ __forceinline__ float strip_bound(float ml, int G, int K, float& gm) {
  switch (G) {
    case 1: return strip_bound_g<1>(ml, K, gm);
    case 2: return strip_bound_g<2>(ml, K, gm);
    case 4: return strip_bound_g<4>(ml, K, gm);
    case 8: return strip_bound_g<8>(ml, K, gm);
    case 16: return strip_bound_g<16>(ml, K, gm);
    default: return strip_bound_g<32>(ml, K, gm);
  }
}

// Order keys of the values a strip or chunk compares, so that a threshold found by bisection
// converts to the compared type exactly: the 16-bit patterns for 16-bit logits compared as
// they are (PACKED), the fp32 patterns otherwise (x = logit + bias in fp32).
template <int DT, bool PACKED>
struct OrderKey {
  static __device__ __forceinline__ uint32_t of(float x) {
    if constexpr (PACKED) {
      uint32_t h;
      if constexpr (DT == DT_F16)
        h = __half_as_ushort(__float2half_rn(x));
      else
        h = __bfloat16_as_ushort(__float2bfloat16_rn(x));
      return (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
    } else {
      return float_ord(x);
    }
  }
  static __device__ __forceinline__ float val(uint32_t k) {
    if constexpr (PACKED) {
      const unsigned short h = (unsigned short)((k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu));
      if constexpr (DT == DT_F16)
        return __half2float(__ushort_as_half(h));
      else
        return __bfloat162float(__ushort_as_bfloat16(h));
    } else {
      return ord_float(k);
    }
  }
};

}  // namespace lsb
