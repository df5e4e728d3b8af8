// Device helpers: inline PTX for mbarriers, bulk (TMA) copies, timers, and the
// order-preserving float keys used by the fine rank.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace lsb {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Test the phase; the warp may be suspended for up to hint_ns while the phase is still
// open (it resumes as soon as the phase completes), so a wait does not spin.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Non-blocking test of the phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the barrier phase with the given parity; give up after limit_ns (a limit of 0
// gives up at once unless the phase is already complete).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  if (limit_ns <= 0) return false;
  const uint32_t hint = limit_ns < 100000 ? (uint32_t)limit_ns : 100000u;
  if (mbar_try_wait(bar, parity, hint)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity, hint)) return true;
    if ((long long)(global_timer_ns() - t0) > limit_ns) return false;
  }
}

// Wait for the phase like mbar_wait_bounded, sleeping sleep_ns between polls: for waits
// that can last microseconds (a pipeline stage, a whole tile), so that a waiting thread does
// not take issue slots from the warps of its SM doing the work.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, long long limit_ns,
                                                uint32_t sleep_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  if (limit_ns <= 0) return false;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    __nanosleep(sleep_ns);
    if (mbar_test_wait(bar, parity)) return true;
    if ((n & 15u) == 0 && (long long)(global_timer_ns() - t0) > limit_ns) return false;
  }
}

// L2 policy: the logits are read exactly once, so let them leave L2 first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Prefetch of `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2; no
// completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only, with an L2 cache policy), in the
// executing thread's current group; completed and visible to that thread after
// cp_async_wait.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's most recent groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 1-D bulk copy global -> shared without an L2 hint (same alignment rules as bulk_load).
__device__ __forceinline__ void bulk_load_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 1-D bulk copy shared -> global (16-byte aligned addresses, size a multiple of 16), in the
// executing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N bulk groups of this thread are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// The rescored candidate beam_score + x - lse in fp32 arithmetic only (FP64 runs at a small
// fraction of the fp32 rate on this part): c = beam_score - lse is kept as an unevaluated pair
// hi + lo of floats (error-free sums, Knuth's two-sum), and hi + x + lo is rounded once more,
// so the score is within about one ulp of the exact value.
struct ScoreBase {
  float hi, lo;
};
__device__ __forceinline__ float2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return make_float2(s, err);
}
// beam_score - (M + log_s), the row's lse being M + log(S); -inf when either is -inf
__device__ __forceinline__ ScoreBase score_base(float beam, float M, float log_s) {
  const float2 a = two_sum(beam, -M);
  const float2 b = two_sum(a.x, -log_s);
  ScoreBase c;
  c.hi = b.x;
  c.lo = __fadd_rn(a.y, b.y);
  if (!isfinite(c.hi)) {
    c.hi = -INFINITY;
    c.lo = 0.0f;
  }
  return c;
}
__device__ __forceinline__ float score_of(const ScoreBase& c, float x) {
  const float2 t = two_sum(c.hi, x);
  if (!isfinite(t.x)) return c.hi == -INFINITY ? -INFINITY : t.x;
  return __fadd_rn(t.x, __fadd_rn(t.y, c.lo));
}

// q = n / d for n < 2^31 with a multiplier prepared on the host (Granlund & Montgomery,
// "Division by invariant integers using multiplication", 1994, round-up variant).
__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint32_t magic, int shift) {
  return (__umulhi(n, magic) + n) >> shift;
}

// Order-preserving map of a float onto uint32 (ascending).  -0 is folded onto +0.
__device__ __forceinline__ uint32_t float_ord(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_float(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

// Key of one candidate for the fine rank; the smaller key ranks first.
// Order: score descending, then parent beam ascending, then logit descending,
// then token id ascending.  For a score of -inf the logit is left out (all such
// candidates are an exact tie broken by the flattened index).
struct Key {
  unsigned long long hi;  // ~ord(score) << 32 | parent
  unsigned long long lo;  // ~ord(x) << 32 | token   (x part zero when score is -inf)
};

__device__ __forceinline__ Key make_key(float s, int parent, float x, int token) {
  Key k;
  const uint32_t so = ~float_ord(s);
  const uint32_t xo = (s == -INFINITY) ? 0u : ~float_ord(x);
  k.hi = ((unsigned long long)so << 32) | (uint32_t)parent;
  k.lo = ((unsigned long long)xo << 32) | (uint32_t)token;
  return k;
}
// Written without short-circuit operators: a branch per comparison costs several times
// the comparison itself in the fine rank's loops.
__device__ __forceinline__ bool key_less(const Key& a, const Key& b) {
  return (a.hi < b.hi) | ((a.hi == b.hi) & (a.lo < b.lo));
}
__device__ __forceinline__ float key_score(const Key& k) { return ord_float(~(uint32_t)(k.hi >> 32)); }
__device__ __forceinline__ int key_parent(const Key& k) { return (int)(uint32_t)(k.hi & 0xffffffffu); }
__device__ __forceinline__ int key_token(const Key& k) { return (int)(uint32_t)(k.lo & 0xffffffffu); }

}  // namespace lsb
