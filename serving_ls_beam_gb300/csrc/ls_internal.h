// Internal definitions shared by the host entry points (api.cu) and the kernels.
// Nothing here is part of the public interface (include/ls_beam.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ls_beam.h"

namespace lsb {

// ---------------------------------------------------------------- kernel shape constants
// K1 (beam_rows.cu): CTAs of kRowWarps independent warps; a warp owns one chunk of
// 32 x VPL 16-byte vectors at a time, streamed through its own 2-stage shared ring.
constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowListOff = 128;   // per-warp mbarriers in [0, 128), then per-warp item lists
constexpr int kRowBarBytes = kRowListOff + kRowWarps * 32 * 4;  // start of the stage buffers
constexpr int kVplMin = 4;         // smallest vectors-per-lane variant built
// K1s (beam_strips.cu): CTAs of kStWarps independent warps; a warp streams one strip of a
// beam's row at a time through its own ring of `stages` stage buffers (at most
// kStMaxStages) and keeps the strip's candidates in a list of kStListCap entries.
constexpr int kStThreads = 256;
constexpr int kStWarps = kStThreads / 32;
constexpr int kStMaxStages = 8;
constexpr int kStListCap = 64;
constexpr int kStTighten = 24;   // candidates of one stage above which the bound is tightened
constexpr int kStListOff = 512;  // per-warp mbarriers in [0, 512), then the per-warp lists
constexpr int kStBarBytes = kStListOff + kStWarps * kStListCap * 8;  // start of the stage buffers
// K3 (beam_fused.cu): one CTA of kFuThreads threads per batch, one warp per strip of a row
// (k * strips per row <= warps), k <= kFuMaxK, at most kFuMaxStages stages per strip (their
// block maxima are kept in shared memory).
constexpr int kFuThreads = 256;
constexpr int kFuMaxK = 8;
constexpr int kFuMaxStages = 32;
constexpr int kFuSampRows = 4;  // rows per CTA of the one-kernel sampler
// K2 (beam_select.cu): one CTA per batch.
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxK = 64;
constexpr int kSelCap = 512;  // survivors the fine rank holds in shared memory
constexpr int kSelStageMax = 96 * 1024;  // a batch's candidate slots staged in shared memory (bytes)

// K0 (logits_rows.cu): the output projection fused with the first traversal; tiles of
// kLgM rows x one chunk (one chunk record per row) of 1 to kLgMaxSubPerChunk sub-tiles of
// kLgN columns, kLgBK of the hidden size per pipeline stage.
constexpr int kLgM = 128;
constexpr int kLgN = 256;
constexpr int kLgMaxSubPerChunk = 4;
constexpr int kLgBK = 64;
constexpr int kLgSwizzleBytes = kLgBK * 2;  // a stage row of kLgBK 16-bit elements is one swizzle row
constexpr int kLgThreads = 192;
constexpr int kLgMaxK = 32;

// Backtrack (backtrack.cu): one CTA per batch, the history staged kBtTileElems entries of
// (token, parent) at a time: 3 x 4 x kBtTileElems = 48 KB of shared memory at most.
constexpr int kBtThreads = 128;
constexpr int kBtTileElems = 4096;

// Device status bits (workspace word 0).
constexpr uint32_t kDevTimeout = 1u << 0;
constexpr uint32_t kDevBadParent = 1u << 1;
constexpr uint32_t kDevInternal = 1u << 2;

// Debug flags (LS_BEAM_DEBUG).
constexpr int kFlagForceExact = 1;
constexpr int kFlagPlainInplace = 2;  // the in-place refresh by the staged CTA kernel
constexpr int kFlagTmaInplace = 32;   // the in-place refresh by bulk copies
constexpr int kFlagWordInplace = 64;  // the in-place refresh by the word kernel (k <= 8)
constexpr int kFlagFusedRefresh = 128;  // ls_beam_step_refresh_inplace in one kernel where K3 applies
constexpr int kFlagChunkRows = 4;     // the beam step's first kernel by fixed-size chunks (K1)
constexpr int kFlagNoFused = 8;       // the beam step as two kernels even where K3 applies
constexpr int kFlagFused = 16;        // the beam step as K3 wherever k allows
constexpr int kFlagNoCluster = 256;   // no cluster form of K3 for small batches (K1s and K2 there)
constexpr int kFlagStaticItems = 2048;  // the bulk-copy refresh without its work counter
constexpr int kFlagCluster = 512;     // the cluster form of K3 wherever k allows, whatever the batch

// ---------------------------------------------------------------- workspace layout
struct alignas(16) RowStat {
  float lse;
  float rtopk;
  int32_t ncand;
  int32_t pad;
};

struct CandSlot {
  float x;    // logit (+ bias) of the candidate
  int32_t v;  // token id within the row
};

struct WsLayout {
  size_t status_off, done_off, rec_off, slot_off, rowstat_off, bstat_off, total;
  int nc_max;      // most chunks per row any plan may use
  int groups;      // G: number of R-top-k groups (power of two >= k)
  int slot_cap;    // C: candidate slots per chunk
  int rec_stride;  // bytes per chunk record
};

__host__ __device__ inline int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Granlund-Montgomery round-up multiplier for division by d (1 <= d < 2^31); the device
// side is fast_div() in ls_device.cuh.  Exact for dividends below 2^31.
inline void make_divisor(uint32_t d, uint32_t* magic, int* shift) {
  int s = 0;
  while ((1ull << s) < d) ++s;
  const unsigned long long m = ((1ull << 32) * ((1ull << s) - d)) / d + 1;
  *magic = (uint32_t)m;
  *shift = s;
}

// Layout for `rows` rows of logits, `nb` per-batch entries and k (the number of top
// elements a row's bound must keep).
inline WsLayout ws_layout_rows(size_t rows, size_t nb, int k, int vocab) {
  WsLayout w{};
  w.groups = pow2_ceil(k);
  w.slot_cap = (int)align_up((size_t)(4 * k + 32), 8);
  w.rec_stride = (int)align_up((size_t)(16 + 4 * w.groups), 16);
  // chunks of 32 x kVplMin vectors over a row of up to 4-byte elements (+ 15 bytes of lead)
  const long long nv_max = (15 + 4ll * vocab + 15) / 16;
  w.nc_max = (int)((nv_max + 32 * kVplMin - 1) / (32 * kVplMin));
  size_t off = 0;
  w.status_off = off;
  off += 256;
  w.done_off = off;
  off = align_up(off + nb * 4, 256);
  w.rec_off = off;
  off = align_up(off + rows * w.nc_max * w.rec_stride, 256);
  w.slot_off = off;
  off = align_up(off + rows * w.nc_max * w.slot_cap * sizeof(CandSlot), 256);
  w.rowstat_off = off;
  off = align_up(off + rows * sizeof(RowStat), 256);
  w.bstat_off = off;
  off = align_up(off + nb * 4, 256);
  w.total = off;
  return w;
}

// Beam step: batch * k rows, one entry per batch.  Returns total == 0 for unsupported shapes.
inline WsLayout ws_layout(int batch, int k, int vocab) {
  if (batch < 0 || k < 1 || k > kMaxK || vocab < k) return WsLayout{};
  return ws_layout_rows((size_t)batch * (size_t)k, (size_t)batch, k, vocab);
}

// Sampling: one row per sequence, top_k kept per row.
inline WsLayout ws_layout_sample(int rows, int top_k, int vocab) {
  if (rows < 0 || top_k < 1 || top_k > kMaxK || vocab < top_k) return WsLayout{};
  return ws_layout_rows((size_t)rows, (size_t)rows, top_k, vocab);
}

// ---------------------------------------------------------------- kernel parameters
struct StepParams {
  const void* logits;
  const float* bias;
  const float* beam;
  const uint8_t* finished;
  int32_t* out_token;
  int32_t* out_parent;
  float* out_score;
  uint8_t* out_finished;
  uint32_t* status;
  uint32_t* done;
  unsigned char* rec;
  CandSlot* slots;
  RowStat* rowstat;
  int32_t* bstat;
  int batch, k, vocab, eos;
  int rows;
  int nc;         // chunks per row
  uint32_t nc_magic;  // fast division by nc
  int nc_shift;
  int groups;
  int slot_cap;
  int rec_stride;
  int flags;
  int sel_stage_bytes;  // K2: bytes of a batch's slots copied to shared memory, 0 = read in place
  int stages;           // K1s: stage buffers per warp
  long long units;  // rows * nc
  long long spin_limit_ns;
  // K3 followed, in the same CTA, by the in-place cache refresh of its batch (the cache
  // [layers, batch * k, heads, max_len, head_dim] by the batch's new parents, positions
  // [0, len)); rf_cache == nullptr: no refresh.  An item is heads [h0, h0 + rf_hg) of one
  // layer and one tile of rf_tile bytes of their slabs.
  unsigned char* rf_cache;
  long long rf_layer_stride, rf_row_stride, rf_slab_stride, rf_slab_bytes;
  int rf_layers, rf_heads, rf_tile, rf_hg;
  // K3 as the one-kernel sampler (sampling decoding): rows are independent sequences, kFuSampRows
  // per CTA, k = top_k; the draw at u[row] writes out_token[row] and out_logprob[row]
  const float* u;
  float* out_logprob;
  float top_p;
};

struct LogitsParams {
  StepParams s;    // workspace, shapes and flags shared with the fine rank (logits unused)
  uint32_t idesc;  // tcgen05 instruction descriptor (operand type, tile shape)
  int dim;         // hidden size
  int n_mp;        // pairs of kLgM-row blocks (one pair per cluster of two CTAs)
  int sub_per_chunk;  // kLgN-column sub-tiles per chunk
  int sub_per_row;    // ceil(vocab / kLgN)
  int n_tiles;     // n_mp * nc
};

struct ReorderParams {
  const unsigned char* src;
  unsigned char* dst;
  const int32_t* parent;
  uint32_t* status;  // may be null
  long long slab_stride;  // bytes between consecutive (l, row, h) slabs = max_len * head_dim * es
  long long row_stride;   // bytes between rows = heads * slab_stride
  long long layer_stride; // bytes between layers = rows * row_stride
  int rows, k, heads, layers;
  int slab_units;   // copy units (of UNIT bytes) per slab = len * head_dim * es / UNIT
  uint32_t div_units_magic;  // fast division by slab_units
  int div_units_shift;
  long long pairs;  // layers * rows
};

struct BacktrackParams {
  const int32_t* tok;  // [steps, batch, k]
  const int32_t* par;  // [steps, batch, k]
  int32_t* seq;        // [batch, k, steps]
  int32_t* len;        // [batch, k]
  uint32_t* status;    // may be null
  int steps, batch, k, eos;
  int tile;            // steps staged per round
};

struct SampleParams {
  const unsigned char* rec;  // K1's chunk records and slots of the rows
  const CandSlot* slots;
  const void* logits;        // [rows, vocab] (exact fallback)
  const float* bias;
  const float* u;            // [rows] uniforms in [0, 1)
  int32_t* out_token;
  float* out_logprob;        // may be null
  RowStat* rowstat;
  int32_t* bstat;
  int rows, vocab, k, nc, groups, slot_cap, rec_stride, flags;
  float top_p;
};

// In-place cache refresh (cache_inplace.cu): staging space per CTA of the plain kernel, per
// stage of the bulk-copy kernel (two stages), and the parents the bulk-copy kernel stages.
constexpr int kIpStageBytes = 48 * 1024;
constexpr int kIpTmaStage = 32 * 1024;  // bulk-copy kernel: each of its two staging buffers (default)
constexpr int kIpWorkOff = 64;  // byte offset of the bulk-copy kernel's work counter in a workspace
constexpr int kIpTmaMaxParents = 8192;

struct InplaceParams {
  unsigned char* cache;
  const int32_t* parent;  // [batch, k]
  uint32_t* status;       // may be null
  long long spin_limit_ns;  // bounded waits of the bulk-copy kernel
  long long layer_stride, row_stride, slab_stride;  // bytes
  long long slab_bytes;   // len * head_dim * es
  uint32_t* work;         // bulk-copy kernel: {next item, CTAs done}, zero between launches; or null
  int tile_bytes;         // positions staged at a time, in bytes (<= stage / k)
  int heads_per_item;     // bulk-copy kernel: heads of one (layer, batch) moved together
  int stage_bytes;        // bulk-copy kernel: bytes of each of its two staging buffers
  int batch, k, heads, layers;
  long long units;        // layers * batch * heads
  // word kernel: an item is heads [h0, h0 + word_heads) of one (layer, batch); its words are
  // word_heads * slab_words, divided by slab_words with (word_magic, word_shift)
  long long slab_words;   // slab_bytes / word size
  int word_heads;
  uint32_t word_magic;
  int word_shift;
  long long word_items;   // layers * batch * ceil(heads / word_heads)
};

// Launch configuration with programmatic dependent launch: the kernel may be scheduled
// while the previous kernel of the stream finishes; it must call griddepcontrol.wait
// before touching anything that kernel (or any earlier work) writes.
struct PdlLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t stream) : cfg{}, attr{} {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

// Host-side checks of ls_beam_step's arguments other than the workspace (api.cu).
ls_status beam_step_check_args(const void* logits, ls_dtype logit_dtype, const float* bias,
                               const float* beam_scores, const uint8_t* finished, int batch, int k, int vocab,
                               int eos_id, const int32_t* out_token, const int32_t* out_parent,
                               const float* out_score, const uint8_t* out_finished);

// Launchers (defined next to their kernels).
size_t beam_rows_smem_bytes(int vpl);
cudaError_t beam_rows_config(int dtype, bool bias, int vpl, int* occupancy);
cudaError_t launch_beam_rows(const StepParams& p, int dtype, int vpl, int grid, cudaStream_t stream);
cudaError_t launch_beam_select(const StepParams& p, int dtype, cudaStream_t stream);
size_t beam_fused_smem_bytes(int vpl, int sps);
cudaError_t beam_fused_config();  // once per device: the kernels' dynamic shared memory
cudaError_t launch_beam_fused(const StepParams& p, int dtype, cudaStream_t stream);
// the one-kernel sampler: ceil(rows / kFuSampRows) CTAs
cudaError_t launch_sample_fused(const StepParams& p, int dtype, cudaStream_t stream);
// the cluster step: one CTA per row (p.nc = 8 strips), a batch's k CTAs one cluster; k a
// power of two up to kFuMaxK
cudaError_t launch_beam_cluster(const StepParams& p, int dtype, cudaStream_t stream);
// bytes of one of a warp's two refresh buffers in K3 for these logits (its VPL)
int beam_fused_refresh_buffer(int dtype, bool bias);
size_t beam_strips_smem_bytes(int vpl, int stages);
cudaError_t beam_strips_config(int dtype, bool bias, int vpl, int stages, int* occupancy);
cudaError_t launch_beam_strips(const StepParams& p, int dtype, int vpl, int grid, cudaStream_t stream);
size_t logits_rows_smem_bytes();
int logits_rows_max_clusters();  // co-resident clusters of two K0 CTAs (0 on error)
cudaError_t logits_rows_config();  // once per device: the kernels' dynamic shared memory
cudaError_t launch_logits_rows(const CUtensorMap& mh, const CUtensorMap& mw, const LogitsParams& lp, int grid,
                               cudaStream_t stream);
cudaError_t beam_select_config();  // once per device: allow kSelStageMax of dynamic shared memory
cudaError_t launch_cache_reorder(const ReorderParams& p, int unit, int grid, cudaStream_t stream);
cudaError_t cache_reorder_occupancy(int unit, int* occupancy);
int backtrack_tile(int k, int steps);
size_t backtrack_smem_bytes(int k, int tile);
cudaError_t launch_backtrack(const BacktrackParams& p, cudaStream_t stream);
cudaError_t launch_sample_select(const SampleParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_cache_inplace(const InplaceParams& p, int unit, int grid, cudaStream_t stream);
cudaError_t cache_inplace_occupancy(int unit, int* occupancy);
// word kernel (k <= kIpWordMaxK): a warp per item, each lane owning word positions
constexpr int kIpWordMaxK = 8;
constexpr int kIpWordThreads = 256;
cudaError_t launch_cache_inplace_words(const InplaceParams& p, int unit, int grid, cudaStream_t stream);
// every batch's parents are staged in shared memory: batch * k <= kIpTmaMaxParents
cudaError_t cache_inplace_words_occupancy(int unit, int batch, int k, int* occupancy);
size_t cache_inplace_tma_smem(int stage_bytes, int batch, int k);
cudaError_t launch_cache_inplace_tma(const InplaceParams& p, int grid, cudaStream_t stream);
cudaError_t cache_inplace_tma_occupancy(int stage_bytes, int batch, int k, int* occupancy);

}  // namespace lsb
