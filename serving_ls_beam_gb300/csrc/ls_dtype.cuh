// Logit element types of the beam step: 16-byte vector unpacking and scalar loads.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace lsb {

enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

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

// The kVec values of one 16-byte vector as floats (exact conversion).
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

// Element e of a 16-byte vector replaced by -inf (used to mask bytes outside a row).
template <int DT>
__device__ __forceinline__ void set_neg_inf(uint4& d, int e) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&d);
  if constexpr (DT == DT_F32) {
    w[e] = Traits<DT>::kNegInfWord;
  } else {
    const uint32_t half = Traits<DT>::kNegInfWord & 0xffffu;
    w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000ffffu) | (half << 16)) : ((w[e >> 1] & 0xffff0000u) | half);
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

// Programmatic dependent launch: wait for the preceding grid's memory / let the next grid launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace lsb
