// End of a search: the token sequence of every final beam, read back through the per-step
// parent pointers of the decode loop's history.
//
// Method: LightSeq inference article (31duo.com, itemid-283120), decoding section: every
// step keeps, for each new beam, the beam it continued (the same parent index that drives
// the cache refresh); a finished hypothesis is read back along those pointers.
//
// GB300 design: one CTA per batch.  Following a parent pointer through global memory costs
// an L2 round trip per step, so the batch's history is staged in shared memory a tile of
// steps at a time (one round of independent coalesced loads per tile), the k walks run in
// shared memory, and the tile's sequences are written back coalesced.
#include "ls_internal.h"

namespace lsb {
namespace {

__global__ void __launch_bounds__(kBtThreads) backtrack_kernel(const BacktrackParams p) {
  extern __shared__ int32_t bt_smem[];
  const int b = blockIdx.x, K = p.k, S = p.tile, tid = threadIdx.x;
  int32_t* tok_s = bt_smem;          // [S][K] tokens of the tile's steps
  int32_t* par_s = tok_s + S * K;    // [S][K] parents
  int32_t* out_s = par_s + S * K;    // [K][S] the tile's part of every sequence
  int c = tid;                       // walker tid follows final beam tid
  int first_eos = p.steps;
  bool bad = false;
  for (int t_hi = p.steps; t_hi > 0; t_hi -= S) {
    const int t_lo = max(0, t_hi - S), n = t_hi - t_lo;
    __syncthreads();  // the previous tile's sequences are written out
    for (int i = tid; i < n * K; i += kBtThreads) {
      const int tt = i / K, j = i - tt * K;
      const size_t h = ((size_t)(t_lo + tt) * p.batch + b) * K + j;
      tok_s[i] = __ldg(p.tok + h);
      par_s[i] = __ldg(p.par + h);
    }
    __syncthreads();
    if (tid < K) {
      for (int tt = n - 1; tt >= 0; --tt) {
        const int cc = min(max(c, 0), K - 1);  // a bad parent is recorded, the walk stays in bounds
        bad |= (c != cc);
        const int tk = tok_s[tt * K + cc];
        out_s[tid * S + tt] = tk;
        first_eos = (tk == p.eos) ? t_lo + tt : first_eos;
        c = par_s[tt * K + cc];
      }
    }
    __syncthreads();
    for (int i = tid; i < K * n; i += kBtThreads) {
      const int j = i / n, tt = i - j * n;
      p.seq[((size_t)b * K + j) * p.steps + t_lo + tt] = out_s[j * S + tt];
    }
  }
  if (tid < K) {
    p.len[(size_t)b * K + tid] = first_eos < p.steps ? first_eos + 1 : p.steps;
    if (bad && p.status) atomicOr(p.status, kDevBadParent);
  }
}

}  // namespace

int backtrack_tile(int k, int steps) {
  const int t = kBtTileElems / k;
  return t < steps ? t : steps;
}

size_t backtrack_smem_bytes(int k, int tile) { return (size_t)3 * tile * k * sizeof(int32_t); }

cudaError_t launch_backtrack(const BacktrackParams& p, cudaStream_t stream) {
  backtrack_kernel<<<p.batch, kBtThreads, backtrack_smem_bytes(p.k, p.tile), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace lsb
