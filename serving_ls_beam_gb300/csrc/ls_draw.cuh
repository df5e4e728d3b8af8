// The draw of sampling decoding, shared by its two kernels (sample.cu after K1, and the
// one-kernel sampler in beam_fused.cu): one warp, one row, from that row's top k candidates
// (tx / tv, best first: larger x, then smaller token).  Probabilities are exp(x - x_0)
// renormalised over the k; below top_p = 1 only the shortest prefix whose cumulative
// probability reaches top_p is kept; the token is the first kept candidate whose cumulative
// probability exceeds u times the kept total.  All in fp32 across the lanes (a prefix sum
// of the k probabilities, then ballots for the cut and the pick), k <= 64.
#pragma once

#include <stdint.h>

namespace lsb {

__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Writes out_token[r] and, when out_logprob is not null, out_logprob[r] = x(token) - lse.
__device__ __forceinline__ void draw_topk(const float* tx, const int* tv, int K, float top_p, float lse, float u,
                                          int r, int32_t* out_token, float* out_logprob) {
  const int lane = threadIdx.x & 31;
  const float x0 = tx[0];
  const float e0 = lane < K ? expf(tx[lane] - x0) : 0.0f;
  const float e1 = lane + 32 < K ? expf(tx[lane + 32] - x0) : 0.0f;
  const float c0 = warp_incl_scan(e0);
  const float t0 = __shfl_sync(0xffffffffu, c0, 31);
  const float c1 = warp_incl_scan(e1) + t0;
  const float tot = __shfl_sync(0xffffffffu, c1, 31);
  int mk = K;  // kept prefix
  if (top_p < 1.0f) {
    const float lim = top_p * tot;
    const unsigned b0 = __ballot_sync(0xffffffffu, (lane < K) & (c0 >= lim));
    const unsigned b1 = __ballot_sync(0xffffffffu, (lane + 32 < K) & (c1 >= lim));
    mk = b0 ? __ffs(b0) : (b1 ? 32 + __ffs(b1) : K);
  }
  const float totm = mk <= 32 ? __shfl_sync(0xffffffffu, c0, mk - 1) : __shfl_sync(0xffffffffu, c1, (mk - 33) & 31);
  const float target = u * totm;
  const unsigned h0 = __ballot_sync(0xffffffffu, (lane < mk) & (c0 > target));
  const unsigned h1 = __ballot_sync(0xffffffffu, (lane + 32 < mk) & (c1 > target));
  const int pick = h0 ? __ffs(h0) - 1 : (h1 ? 31 + __ffs(h1) : mk - 1);
  if (lane == 0) {
    out_token[r] = tv[pick];
    if (out_logprob) out_logprob[r] = tx[pick] - lse;
  }
}

}  // namespace lsb
