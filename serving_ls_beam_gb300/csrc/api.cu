// C-ABI entry points (include/ls_beam.h): argument checks on the host, launch plans,
// and the enqueue of the kernels on the caller's stream.  The library holds no state
// besides per-device properties cached on first use.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ls_beam.h"
#include "ls_internal.h"

using namespace lsb;

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultSpinNs = 2000000000LL;  // 2 s per bounded wait

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  bool select_ready = false;  // K2's dynamic shared-memory limit raised
  bool logits_ready = false;  // K0's dynamic shared-memory limit raised
  bool fused_ready = false;   // K3's dynamic shared-memory limit raised
  int logits_clusters = 0;    // co-resident clusters of two K0 CTAs
  // K1 occupancy per [dtype][bias][vpl index]; 0 = not configured yet
  int step_occ[3][2][3] = {};
  // K1s occupancy per [dtype][bias][stages]
  int strip_occ[3][2][kStMaxStages + 1] = {};
  int copy_occ[5] = {};
  int inplace_occ[5] = {};
  int words_occ[10] = {};  // word kernel per [unit index][k <= 4 or <= 8]
  long long words_parents[10] = {};  // the batch * k that occupancy was computed for
  int inplace_tma_occ = 0;
  size_t inplace_tma_smem = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

int vpl_index(int vpl) { return vpl == 4 ? 0 : (vpl == 8 ? 1 : (vpl == 16 ? 2 : -1)); }
int unit_index(int unit) { return unit == 16 ? 0 : unit == 8 ? 1 : unit == 4 ? 2 : unit == 2 ? 3 : 4; }

struct Debug {
  int flags = 0;
  long long spin_ns = kDefaultSpinNs;
  int vpl = 0;     // 0 = plan's choice
  int stages = 0;  // K1s stage buffers per warp, 0 = plan's choice
  int parts = 0;   // K1s strips per row, 0 = plan's choice
  int ipw = 0;     // in-place word kernel: words per item, 0 = plan's choice
  int ipkeff = 0;  // in-place bulk-copy kernel: parents an item is sized for, 0 = plan's choice
  int ipstage = 0; // in-place bulk-copy kernel: bytes of each staging buffer, 0 = plan's choice
  int stage = -1;  // K2 after K0: 1 = stage the batch's slots, 0 = read them in place, -1 = plan
  bool check_ptrs = true;
};

// LS_BEAM_DEBUG: comma-separated "exact", "ipplain", "iptma", "ipwords", "ipstatic", "steprefresh", "chunk", "strips",
// "fused", "nofused", "cluster", "nocluster", "spin=<ns>", "vpl=<4|8|16>", "stages=<2..8>", "parts=<n>", "ipw=<words>",
// "ipkeff=<parents>", "ipstage=<bytes>", "stage=<0|1>", "nocheck".
Debug read_debug() {
  Debug d;
  const char* env = std::getenv("LS_BEAM_DEBUG");
  if (!env || !*env) return d;
  char buf[256];
  std::strncpy(buf, env, sizeof buf - 1);
  buf[sizeof buf - 1] = 0;
  for (char* tok = std::strtok(buf, ","); tok; tok = std::strtok(nullptr, ",")) {
    if (!std::strcmp(tok, "exact")) d.flags |= kFlagForceExact;
    else if (!std::strcmp(tok, "ipplain")) d.flags |= kFlagPlainInplace;
    else if (!std::strcmp(tok, "iptma")) d.flags |= kFlagTmaInplace;
    else if (!std::strcmp(tok, "ipstatic")) d.flags |= kFlagStaticItems;
    else if (!std::strcmp(tok, "ipwords")) d.flags |= kFlagWordInplace;
    else if (!std::strcmp(tok, "steprefresh")) d.flags |= kFlagFusedRefresh;
    else if (!std::strncmp(tok, "spin=", 5)) d.spin_ns = std::atoll(tok + 5);
    else if (!std::strcmp(tok, "chunk")) d.flags |= kFlagChunkRows;
    else if (!std::strcmp(tok, "strips")) d.flags &= ~kFlagChunkRows;
    else if (!std::strcmp(tok, "fused")) d.flags |= kFlagFused;
    else if (!std::strcmp(tok, "nofused")) d.flags |= kFlagNoFused;
    else if (!std::strcmp(tok, "nocluster")) d.flags |= kFlagNoCluster;
    else if (!std::strcmp(tok, "cluster")) d.flags |= kFlagCluster;
    else if (!std::strncmp(tok, "vpl=", 4)) d.vpl = std::atoi(tok + 4);
    else if (!std::strncmp(tok, "stages=", 7)) d.stages = std::atoi(tok + 7);
    else if (!std::strncmp(tok, "parts=", 6)) d.parts = std::atoi(tok + 6);
    else if (!std::strncmp(tok, "ipw=", 4)) d.ipw = std::atoi(tok + 4);
    else if (!std::strncmp(tok, "ipkeff=", 7)) d.ipkeff = std::atoi(tok + 7);
    else if (!std::strncmp(tok, "ipstage=", 8)) d.ipstage = std::atoi(tok + 8);
    else if (!std::strncmp(tok, "stage=", 6)) d.stage = std::atoi(tok + 6);
    else if (!std::strcmp(tok, "nocheck")) d.check_ptrs = false;
  }
  if (d.spin_ns < 0) d.spin_ns = 0;
  if (vpl_index(d.vpl) < 0) d.vpl = 0;
  if (d.stages < 0 || d.stages > kStMaxStages) d.stages = 0;
  if (d.parts < 0) d.parts = 0;
  return d;
}

ls_status cuda_fail(cudaError_t e) {
  (void)e;
  cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return LS_ERR_CUDA;
}

DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  *dev_out = dev;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    di.ready = true;
  }
  return &di;
}

int step_occupancy(DeviceInfo* di, int dtype, bool bias, int vpl) {
  std::lock_guard<std::mutex> lk(g_mu);
  int& occ = di->step_occ[dtype][bias ? 1 : 0][vpl_index(vpl)];
  if (occ == 0) {
    int o = 0;
    if (beam_rows_config(dtype, bias, vpl, &o) != cudaSuccess || o < 1) return 0;
    occ = o;
  }
  return occ;
}

// K1's launch plan for `rows` rows of `vocab` logits of `es` bytes.
struct RowPlan {
  int vpl, nc;
  long long units, grid;
};

ls_status plan_rows(DeviceInfo* di, const Debug& dbg, int dtype, int es, bool bias, int vocab, long long rows,
                    const WsLayout& wl, RowPlan* out) {
  // 8 vectors per lane (4 KB chunks) unless 16-bit logits with a bias (register pressure)
  const int vpl = dbg.vpl ? dbg.vpl : ((es == 2 && bias) ? 4 : 8);
  const int occ = step_occupancy(di, dtype, bias, vpl);
  if (occ < 1) return cuda_fail(cudaErrorUnknown);
  // a row spans at most ceil((15 + vocab * es) / 16) aligned 16-byte vectors
  const long long nv_max = (15 + (long long)vocab * es + 15) / 16;
  const int cv = 32 * vpl;
  const int nc = (int)((nv_max + cv - 1) / cv);
  if (nc > wl.nc_max) return LS_ERR_INTERNAL;
  out->vpl = vpl;
  out->nc = nc;
  out->units = rows * nc;
  const long long grid_full = (long long)di->sms * occ;
  const long long grid_need = (out->units + kRowWarps - 1) / kRowWarps;
  out->grid = grid_need < grid_full ? grid_need : grid_full;
  return LS_OK;
}

int strip_occupancy(DeviceInfo* di, int dtype, bool bias, int vpl, int stages) {
  std::lock_guard<std::mutex> lk(g_mu);
  int& occ = di->strip_occ[dtype][bias ? 1 : 0][stages];
  if (occ == 0) {
    int o = 0;
    if (beam_strips_config(dtype, bias, vpl, stages, &o) != cudaSuccess || o < 1) return 0;
    occ = o;
  }
  return occ;
}

// K1s's launch plan for `rows` rows of `vocab` logits of `es` bytes: W strips per row (the
// unit count rows * W fits the resident warps once, W at most the stages of the shortest
// row, so every strip has at least one stage), one unit per warp.
struct StripPlan {
  int vpl, stages, parts;
  long long units, grid;
};

ls_status plan_strips(DeviceInfo* di, const Debug& dbg, int dtype, int es, bool bias, int vocab, long long rows,
                      const WsLayout& wl, StripPlan* out) {
  const int vpl = (es == 2 && bias) ? 4 : 8;  // 64 packed or 32 float elements per lane and stage
  const int stages = dbg.stages ? dbg.stages : 2;
  const int occ = strip_occupancy(di, dtype, bias, vpl, stages);
  if (occ < 1) return cuda_fail(cudaErrorUnknown);
  const long long cv = 32ll * vpl;
  const long long ns_min = ((long long)vocab * es / 16 + cv - 1) / cv;  // stages of a 16-byte aligned row
  const long long slots = (long long)di->sms * occ * kStWarps;
  long long w = dbg.parts ? dbg.parts : slots / (rows > 0 ? rows : 1);
  if (w > ns_min) w = ns_min;
  if (w > wl.nc_max) w = wl.nc_max;
  if (w < 1) w = 1;
  out->vpl = vpl;
  out->stages = stages;
  out->parts = (int)w;
  out->units = rows * w;
  const long long grid_full = (long long)di->sms * occ;
  const long long grid_need = (out->units + kStWarps - 1) / kStWarps;
  out->grid = grid_need < grid_full ? grid_need : grid_full;
  return LS_OK;
}

int inplace_occupancy(DeviceInfo* di, int unit) {
  std::lock_guard<std::mutex> lk(g_mu);
  int& occ = di->inplace_occ[unit_index(unit)];
  if (occ == 0) {
    int o = 0;
    if (cache_inplace_occupancy(unit, &o) != cudaSuccess || o < 1) return 0;
    occ = o;
  }
  return occ;
}

// occupancy of the word kernel for (unit, k <= 4 or <= 8), computed once per device
int inplace_words_occupancy(DeviceInfo* di, int unit, int batch, int k) {
  // the shared memory (the parents) varies with batch * k: looked up again when it grows
  std::lock_guard<std::mutex> lk(g_mu);
  const int slot = unit_index(unit) * 2 + (k <= 4 ? 0 : 1);
  int& occ = di->words_occ[slot];
  long long& parents = di->words_parents[slot];
  if (occ == 0 || (long long)batch * k > parents) {
    int o = 0;
    if (cache_inplace_words_occupancy(unit, batch, k, &o) != cudaSuccess || o < 1) return 0;
    occ = o;
    parents = (long long)batch * k;
  }
  return occ;
}

int inplace_tma_occupancy(DeviceInfo* di, int stage_bytes, int batch, int k) {
  std::lock_guard<std::mutex> lk(g_mu);
  const size_t smem = cache_inplace_tma_smem(stage_bytes, batch, k);
  if (di->inplace_tma_occ == 0 || di->inplace_tma_smem != smem) {
    int o = 0;
    if (cache_inplace_tma_occupancy(stage_bytes, batch, k, &o) != cudaSuccess || o < 1) return 0;
    di->inplace_tma_occ = o;
    di->inplace_tma_smem = smem;
  }
  return di->inplace_tma_occ;
}

bool select_configured(DeviceInfo* di) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!di->select_ready) {
    if (beam_select_config() != cudaSuccess) return false;
    di->select_ready = true;
  }
  return true;
}

bool fused_configured(DeviceInfo* di) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!di->fused_ready) {
    if (beam_fused_config() != cudaSuccess) return false;
    di->fused_ready = true;
  }
  return true;
}

bool logits_configured(DeviceInfo* di) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!di->logits_ready) {
    if (logits_rows_config() != cudaSuccess) return false;
    di->logits_clusters = logits_rows_max_clusters();
    di->logits_ready = true;
  }
  return true;
}

int logits_clusters(DeviceInfo* di) {
  std::lock_guard<std::mutex> lk(g_mu);
  return di->logits_clusters;
}

// cuTensorMapEncodeTiled, looked up in the driver once (the library does not link libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map of a row-major [outer, inner] f16 / bf16 matrix read in boxes of kLgBK inner
// elements (kLgSwizzleBytes, one swizzle row) by box_outer rows; reads outside the
// matrix return zeros.
bool encode_kmajor(CUtensorMap* m, const void* base, ls_dtype dt, long long inner, long long outer, int box_outer) {
  const EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kLgBK, (cuuint32_t)box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt == LS_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            kLgSwizzleBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Instruction descriptor of tcgen05.mma kind::f16 for K0's tile: f32 accumulators, A and
// B of the same 16-bit type, both K-major, M = kLgM, N = kLgN.
uint32_t umma_idesc(bool bf16) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(kLgN >> 3) << 17) | ((uint32_t)(kLgM >> 4) << 24);
}

int copy_occupancy(DeviceInfo* di, int unit) {
  std::lock_guard<std::mutex> lk(g_mu);
  int& occ = di->copy_occ[unit_index(unit)];
  if (occ == 0) {
    int o = 0;
    if (cache_reorder_occupancy(unit, &o) != cudaSuccess || o < 1) return 0;
    occ = o;
  }
  return occ;
}

// Device-reachable memory: device, managed, or registered host memory.
bool device_reachable(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int dtype_bytes(ls_dtype d) { return d == LS_DTYPE_F32 ? 4 : 2; }
bool dtype_ok(ls_dtype d) { return d == LS_DTYPE_F32 || d == LS_DTYPE_F16 || d == LS_DTYPE_BF16; }

}  // namespace

extern "C" {

size_t ls_beam_step_workspace_size(int batch, int k, int vocab) {
  if (batch < 0 || k < 1 || k > LS_MAX_K || vocab < k) return 0;
  if ((long long)k * vocab >= (1ll << 31) || vocab > (1 << 28)) return 0;
  if ((long long)batch * k * ws_layout(batch, k, vocab).nc_max >= (1ll << 31)) return 0;
  return ws_layout(batch, k, vocab).total;
}

ls_status ls_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes == 0) return LS_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

}  // extern "C"

namespace lsb {

// The host-side checks of ls_beam_step's arguments other than the workspace: LS_OK when they
// pass (batch == 0 included), LS_ERR_INVALID_ARG otherwise.
ls_status beam_step_check_args(const void* logits, ls_dtype logit_dtype, const float* bias,
                               const float* beam_scores, const uint8_t* finished, int batch, int k, int vocab,
                               int eos_id, const int32_t* out_token, const int32_t* out_parent,
                               const float* out_score, const uint8_t* out_finished) {
  if (batch < 0 || k < 1 || k > LS_MAX_K || vocab < k) return LS_ERR_INVALID_ARG;
  if ((long long)k * vocab >= (1ll << 31) || vocab > (1 << 28)) return LS_ERR_INVALID_ARG;
  if (eos_id < 0 || eos_id >= vocab) return LS_ERR_INVALID_ARG;
  if (!dtype_ok(logit_dtype)) return LS_ERR_INVALID_ARG;
  if (batch == 0) return LS_OK;
  if (!logits || !beam_scores || !out_token || !out_parent || !out_score) return LS_ERR_INVALID_ARG;
  const int es = dtype_bytes(logit_dtype);
  if (!aligned(logits, es) || (bias && !aligned(bias, 4)) || !aligned(beam_scores, 4) || !aligned(out_token, 4) ||
      !aligned(out_parent, 4) || !aligned(out_score, 4))
    return LS_ERR_INVALID_ARG;
  if (read_debug().check_ptrs) {
    const void* ptrs[] = {logits, bias, beam_scores, finished, out_token, out_parent, out_score, out_finished};
    for (const void* q : ptrs)
      if (q && !device_reachable(q)) return LS_ERR_INVALID_ARG;
  }
  return LS_OK;
}

// The argument checks of ls_cache_refresh_inplace (an empty shape passes).
ls_status inplace_check_args(void* cache, ls_dtype dtype, const int32_t* parent, int layers, int batch, int k,
                             int heads, int max_len, int len, int head_dim, void* workspace) {
  if (layers < 0 || batch < 0 || k < 1 || k > LS_MAX_K || heads < 0 || max_len < 0 || len < 0 || len > max_len ||
      head_dim < 0)
    return LS_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return LS_ERR_INVALID_ARG;
  if (layers == 0 || batch == 0 || heads == 0 || len == 0 || head_dim == 0) return LS_OK;
  if (!cache || !parent) return LS_ERR_INVALID_ARG;
  if (!aligned(parent, 4) || (workspace && !aligned(workspace, 256))) return LS_ERR_INVALID_ARG;
  if (read_debug().check_ptrs) {
    if (!device_reachable(cache) || !device_reachable(parent)) return LS_ERR_INVALID_ARG;
    if (workspace && !device_reachable(workspace)) return LS_ERR_INVALID_ARG;
  }
  return LS_OK;
}

}  // namespace lsb

extern "C" {

// The in-place cache refresh a step may run in its own kernel (K3), as the host planned it.
struct FusedRefresh {
  unsigned char* cache;
  int es;  // element size of the cache
  int layers, heads, max_len, len, head_dim;
};

// ls_beam_step; with rf != nullptr, K3 also refreshes the cache when its plan is taken and
// the cache suits the bulk copies (*refreshed is set then).
static ls_status beam_step_impl(const void* logits, ls_dtype logit_dtype, const float* bias, const float* beam_scores,
                         const uint8_t* finished, int batch, int k, int vocab, int eos_id, int32_t* out_token,
                         int32_t* out_parent, float* out_score, uint8_t* out_finished, void* workspace,
                         size_t workspace_bytes, void* stream, const FusedRefresh* rf, bool* refreshed) {
  if (refreshed) *refreshed = false;
  const ls_status chk = beam_step_check_args(logits, logit_dtype, bias, beam_scores, finished, batch, k, vocab,
                                             eos_id, out_token, out_parent, out_score, out_finished);
  if (chk != LS_OK || batch == 0) return chk;
  if (!workspace) return LS_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(batch, k, vocab);
  if (wl.total == 0 || workspace_bytes < wl.total) return LS_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return LS_ERR_INVALID_ARG;
  const Debug dbg = read_debug();
  if (dbg.check_ptrs && !device_reachable(workspace)) return LS_ERR_INVALID_ARG;
  const int es = dtype_bytes(logit_dtype);
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (!di) return cuda_fail(cudaErrorUnknown);

  const int dtype = (int)logit_dtype;
  const long long rows = (long long)batch * k;
  // K3 (the whole step of a batch in one CTA) when the batches fill the GPU by themselves, or
  // when the rows are more than the cluster form runs in one wave (two CTAs per SM), and every
  // strip's block maxima fit its shared memory
  int fu_parts = (kFuThreads / 32) / k;
  if (dbg.parts > 0 && dbg.parts * k <= kFuThreads / 32) fu_parts = dbg.parts;
  const int fu_vpl = (dtype == LS_DTYPE_F32 || bias) ? 4 : 8;
  const long long fu_ns = ((15 + (long long)vocab * es + 15) / 16 + 32ll * fu_vpl - 1) / (32ll * fu_vpl);
  const bool fused = !(dbg.flags & kFlagNoFused) && k <= kFuMaxK && fu_parts >= 1 &&
                     (fu_ns + fu_parts - 1) / fu_parts <= kFuMaxStages &&
                     ((dbg.flags & kFlagFused) || 2ll * batch >= di->sms || rows > 2ll * di->sms);
  // otherwise K3's cluster form for k a power of two up to 8 (a CTA of eight strips per row, a
  // batch's k CTAs one cluster) when the rows are at least a third of the SMs; fewer rows take
  // the two-kernel path, whose strips spread a row over more warps.  One launch, f16 unless
  // noted: 64 x 8 x 40000 K3 26.6 us, cluster 36.9 (two waves); 32 x 8 x 40000 cluster 22.5,
  // K3 26.6, two kernels 32.8; 8 x 8 x 120000 f32 cluster 25.2, two kernels 41.6; 8 x 4 x 250000
  // two kernels 22.6, cluster 24.6; 8 x 1 x 50257 two kernels 12.3, cluster 14.3
  constexpr int kClParts = kFuThreads / 32;
  const bool cluster = (!fused || (dbg.flags & kFlagCluster)) && !(dbg.flags & (kFlagNoFused | kFlagNoCluster)) &&
                       k <= kFuMaxK && (k & (k - 1)) == 0 && (fu_ns + kClParts - 1) / kClParts <= kFuMaxStages &&
                       ((dbg.flags & kFlagCluster) || 3ll * rows >= di->sms);
  if (fused || cluster) {
    if (!fused_configured(di)) return cuda_fail(cudaErrorUnknown);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    StepParams p = {};
    p.logits = logits;
    p.bias = bias;
    p.beam = beam_scores;
    p.finished = finished;
    p.out_token = out_token;
    p.out_parent = out_parent;
    p.out_score = out_score;
    p.out_finished = out_finished;
    p.status = reinterpret_cast<uint32_t*>(ws + wl.status_off);
    p.rowstat = reinterpret_cast<RowStat*>(ws + wl.rowstat_off);
    p.bstat = reinterpret_cast<int32_t*>(ws + wl.bstat_off);
    p.batch = batch;
    p.k = k;
    p.vocab = vocab;
    p.eos = eos_id;
    p.rows = (int)rows;
    const int parts = cluster ? kClParts : fu_parts;
    p.nc = parts;                                    // strips per row, one warp each
    p.stages = (int)((fu_ns + parts - 1) / parts);  // block-max rows per strip
    p.flags = dbg.flags;
    p.spin_limit_ns = dbg.spin_ns;
    if (cluster) {
      const cudaError_t e = launch_beam_cluster(p, dtype, static_cast<cudaStream_t>(stream));
      return e == cudaSuccess ? LS_OK : cuda_fail(e);
    }
    if (rf && (dbg.flags & kFlagFusedRefresh)) {
      // the batch's refresh in K3: bulk copies of 16-byte aligned slabs through two buffers
      // per warp; a tile of a slab (positions) per parent, or several heads' whole slabs
      const long long slab_stride = (long long)rf->max_len * rf->head_dim * rf->es;
      const long long slab_bytes = (long long)rf->len * rf->head_dim * rf->es;
      const long long buf = beam_fused_refresh_buffer(dtype, bias != nullptr);
      long long tile = (buf / k) / 16 * 16;
      const bool fits = aligned(rf->cache, 16) && slab_stride % 16 == 0 && slab_bytes % 16 == 0 && tile >= 16;
      if (fits) {
        long long hg = 1;
        if (slab_bytes <= tile) {
          tile = slab_bytes;
          hg = buf / ((long long)k * slab_bytes);
          hg = hg < 1 ? 1 : (hg > rf->heads ? rf->heads : hg);
        }
        p.rf_cache = rf->cache;
        p.rf_slab_stride = slab_stride;
        p.rf_row_stride = slab_stride * rf->heads;
        p.rf_layer_stride = p.rf_row_stride * rows;
        p.rf_slab_bytes = slab_bytes;
        p.rf_layers = rf->layers;
        p.rf_heads = rf->heads;
        p.rf_tile = (int)tile;
        p.rf_hg = (int)hg;
        if (refreshed) *refreshed = true;
      }
    }
    const cudaError_t e = launch_beam_fused(p, dtype, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LS_OK : cuda_fail(e);
  }
  // K1s (a warp streams a strip of a row) unless forced to K1 (fixed-size chunks); K1s
  // holds the group maxima in lanes, so k <= 32
  const bool strips = !(dbg.flags & kFlagChunkRows) && k <= 32;
  RowPlan plan{};
  StripPlan splan{};
  const ls_status ps = strips ? plan_strips(di, dbg, dtype, es, bias != nullptr, vocab, rows, wl, &splan)
                              : plan_rows(di, dbg, dtype, es, bias != nullptr, vocab, rows, wl, &plan);
  if (ps != LS_OK) return ps;
  const int vpl = strips ? splan.vpl : plan.vpl, nc = strips ? splan.parts : plan.nc;
  const long long units = strips ? splan.units : plan.units, grid = strips ? splan.grid : plan.grid;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  StepParams p;
  p.logits = logits;
  p.bias = bias;
  p.beam = beam_scores;
  p.finished = finished;
  p.out_token = out_token;
  p.out_parent = out_parent;
  p.out_score = out_score;
  p.out_finished = out_finished;
  p.status = reinterpret_cast<uint32_t*>(ws + wl.status_off);
  p.done = reinterpret_cast<uint32_t*>(ws + wl.done_off);
  p.rec = ws + wl.rec_off;
  p.slots = reinterpret_cast<CandSlot*>(ws + wl.slot_off);
  p.rowstat = reinterpret_cast<RowStat*>(ws + wl.rowstat_off);
  p.bstat = reinterpret_cast<int32_t*>(ws + wl.bstat_off);
  p.batch = batch;
  p.k = k;
  p.vocab = vocab;
  p.eos = eos_id;
  p.rows = (int)rows;
  p.nc = nc;
  make_divisor((uint32_t)nc, &p.nc_magic, &p.nc_shift);
  p.groups = wl.groups;
  p.slot_cap = wl.slot_cap;
  p.rec_stride = wl.rec_stride;
  p.flags = dbg.flags;
  // K2 copies a batch's slots to shared memory in one bulk copy when they fit (k <= 8)
  const long long stage = (long long)k * nc * wl.slot_cap * (long long)sizeof(CandSlot);
  p.sel_stage_bytes = (k <= 8 && nc <= 128 && (long long)k * nc <= 1024 && stage <= kSelStageMax) ? (int)stage : 0;
  if (!select_configured(di)) return cuda_fail(cudaErrorUnknown);
  p.units = units;
  p.spin_limit_ns = dbg.spin_ns;
  p.stages = splan.stages;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = strips ? launch_beam_strips(p, dtype, vpl, (int)grid, st) : launch_beam_rows(p, dtype, vpl, (int)grid, st);
  if (e == cudaSuccess) e = launch_beam_select(p, dtype, st);
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

ls_status ls_beam_step(const void* logits, ls_dtype logit_dtype, const float* bias, const float* beam_scores,
                       const uint8_t* finished, int batch, int k, int vocab, int eos_id, int32_t* out_token,
                       int32_t* out_parent, float* out_score, uint8_t* out_finished, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return beam_step_impl(logits, logit_dtype, bias, beam_scores, finished, batch, k, vocab, eos_id, out_token,
                        out_parent, out_score, out_finished, workspace, workspace_bytes, stream, nullptr, nullptr);
}

ls_status ls_beam_step_refresh_inplace(const void* logits, ls_dtype logit_dtype, const float* bias,
                                       const float* beam_scores, const uint8_t* finished, int batch, int k,
                                       int vocab, int eos_id, int32_t* out_token, int32_t* out_parent,
                                       float* out_score, uint8_t* out_finished, void* cache, ls_dtype cache_dtype,
                                       int layers, int heads, int max_len, int len, int head_dim, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  // every argument of both calls is checked before anything is queued
  if (!out_parent) return LS_ERR_INVALID_ARG;
  const ls_status ci = inplace_check_args(cache, cache_dtype, out_parent, layers, batch, k, heads, max_len, len,
                                          head_dim, workspace);
  if (ci != LS_OK) return ci;
  const bool empty_cache = layers == 0 || batch == 0 || heads == 0 || len == 0 || head_dim == 0;
  FusedRefresh rf{static_cast<unsigned char*>(cache), dtype_bytes(cache_dtype), layers, heads, max_len, len,
                  head_dim};
  bool refreshed = false;
  const ls_status st = beam_step_impl(logits, logit_dtype, bias, beam_scores, finished, batch, k, vocab, eos_id,
                                      out_token, out_parent, out_score, out_finished, workspace, workspace_bytes,
                                      stream, empty_cache ? nullptr : &rf, &refreshed);
  if (st != LS_OK || refreshed || empty_cache) return st;
  return ls_cache_refresh_inplace(cache, cache_dtype, out_parent, layers, batch, k, heads, max_len, len, head_dim,
                                  workspace, stream);
}

ls_status ls_logits_beam_step(const void* hidden, const void* weight, ls_dtype dtype, int dim, const float* bias,
                              const float* beam_scores, const uint8_t* finished, int batch, int k, int vocab,
                              int eos_id, int32_t* out_token, int32_t* out_parent, float* out_score,
                              uint8_t* out_finished, void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || k < 1 || k > LS_MAX_K || vocab < k) return LS_ERR_INVALID_ARG;
  if ((long long)k * vocab >= (1ll << 31) || vocab > (1 << 28)) return LS_ERR_INVALID_ARG;
  if (eos_id < 0 || eos_id >= vocab) return LS_ERR_INVALID_ARG;
  if (dtype != LS_DTYPE_F16 && dtype != LS_DTYPE_BF16) return LS_ERR_INVALID_ARG;
  if (dim < 8 || dim % 8 != 0) return LS_ERR_INVALID_ARG;
  if (k > kLgMaxK) return LS_ERR_UNSUPPORTED;
  if (batch == 0) return LS_OK;
  if (!hidden || !weight || !beam_scores || !out_token || !out_parent || !out_score || !workspace)
    return LS_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout(batch, k, vocab);
  if (wl.total == 0 || workspace_bytes < wl.total) return LS_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || (bias && !aligned(bias, 4)) || !aligned(beam_scores, 4) ||
      !aligned(out_token, 4) || !aligned(out_parent, 4) || !aligned(out_score, 4) || !aligned(workspace, 256))
    return LS_ERR_INVALID_ARG;
  const long long rows = (long long)batch * k;
  if (rows >= (1ll << 31) || rows * dim >= (1ll << 40)) return LS_ERR_UNSUPPORTED;
  const Debug dbg = read_debug();
  if (dbg.check_ptrs) {
    const void* ptrs[] = {hidden, weight, bias, beam_scores, finished, out_token, out_parent, out_score, out_finished,
                          workspace};
    for (const void* q : ptrs)
      if (q && !device_reachable(q)) return LS_ERR_INVALID_ARG;
  }
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (!di) return cuda_fail(cudaErrorUnknown);
  if (!logits_configured(di) || !select_configured(di)) return cuda_fail(cudaErrorUnknown);
  // chunk width: 1 to kLgMaxSubPerChunk sub-tiles, the one whose tiles spread best over the
  // clusters (fewest sub-tiles for the busiest cluster), within the workspace's chunks per
  // row and leaving every sub-tile of a chunk room for k candidates
  const long long n_m = (rows + kLgM - 1) / kLgM;
  const int n_mp = (int)((n_m + 1) / 2);
  const int sub_per_row = (vocab + kLgN - 1) / kLgN;
  const int clusters = logits_clusters(di);
  if (clusters < 1) return cuda_fail(cudaErrorUnknown);
  int spc = 0;
  long long best = 0;
  for (int s = 1; s <= kLgMaxSubPerChunk; ++s) {
    const long long ncs = (sub_per_row + s - 1) / s;
    if (ncs > wl.nc_max || wl.slot_cap - k * (s - 1) < 2 * k) continue;
    const long long rounds = ((long long)n_mp * ncs + clusters - 1) / clusters;
    if (spc == 0 || rounds * s < best) {
      spc = s;
      best = rounds * s;
    }
  }
  if (spc == 0) return LS_ERR_INTERNAL;
  const int nc = (sub_per_row + spc - 1) / spc;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  LogitsParams lp;
  StepParams& p = lp.s;
  p = StepParams{};
  p.logits = nullptr;  // the logits are never stored
  p.bias = bias;
  p.beam = beam_scores;
  p.finished = finished;
  p.out_token = out_token;
  p.out_parent = out_parent;
  p.out_score = out_score;
  p.out_finished = out_finished;
  p.status = reinterpret_cast<uint32_t*>(ws + wl.status_off);
  p.done = reinterpret_cast<uint32_t*>(ws + wl.done_off);
  p.rec = ws + wl.rec_off;
  p.slots = reinterpret_cast<CandSlot*>(ws + wl.slot_off);
  p.rowstat = reinterpret_cast<RowStat*>(ws + wl.rowstat_off);
  p.bstat = reinterpret_cast<int32_t*>(ws + wl.bstat_off);
  p.batch = batch;
  p.k = k;
  p.vocab = vocab;
  p.eos = eos_id;
  p.rows = (int)rows;
  p.nc = nc;
  make_divisor((uint32_t)nc, &p.nc_magic, &p.nc_shift);
  p.groups = wl.groups;
  p.slot_cap = wl.slot_cap;
  p.rec_stride = wl.rec_stride;
  p.flags = dbg.flags;
  const long long stage = (long long)k * nc * wl.slot_cap * (long long)sizeof(CandSlot);
  p.sel_stage_bytes = (k <= 8 && nc <= 128 && (long long)k * nc <= 1024 && stage <= kSelStageMax) ? (int)stage : 0;
  if (dbg.stage == 0) p.sel_stage_bytes = 0;
  p.units = rows * nc;
  p.spin_limit_ns = dbg.spin_ns;
  lp.idesc = umma_idesc(dtype == LS_DTYPE_BF16);
  lp.dim = dim;
  lp.n_mp = n_mp;
  lp.sub_per_chunk = spc;
  lp.sub_per_row = sub_per_row;
  const long long n_tiles = (long long)lp.n_mp * nc;
  if (n_tiles >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  lp.n_tiles = (int)n_tiles;
  const int grid = 2 * (int)(n_tiles < clusters ? n_tiles : clusters);

  CUtensorMap mh, mw;
  if (!encode_kmajor(&mh, hidden, dtype, dim, rows, kLgM) ||
      !encode_kmajor(&mw, weight, dtype, dim, vocab, kLgN))
    return cuda_fail(cudaErrorUnknown);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_logits_rows(mh, mw, lp, grid, st);
  if (e == cudaSuccess) {
    StepParams ps = p;
    ps.bias = nullptr;  // the slots hold x = logit + bias already
    e = launch_beam_select(ps, (int)LS_DTYPE_F32, st);
  }
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

ls_status ls_cache_reorder(const void* src, void* dst, ls_dtype dtype, const int32_t* parent, int layers, int batch,
                           int k, int heads, int max_len, int len, int head_dim, void* workspace, void* stream) {
  if (layers < 0 || batch < 0 || k < 1 || heads < 0 || max_len < 0 || len < 0 || len > max_len || head_dim < 0)
    return LS_ERR_INVALID_ARG;
  if (!dtype_ok(dtype)) return LS_ERR_INVALID_ARG;
  if (layers == 0 || batch == 0 || heads == 0 || len == 0 || head_dim == 0) return LS_OK;
  if (!src || !dst || !parent) return LS_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return LS_ERR_INVALID_ARG;
  const long long es = dtype_bytes(dtype);
  const long long rows = (long long)batch * k;
  const long long slab_stride = (long long)max_len * head_dim * es;
  const long long row_stride = slab_stride * heads;
  const long long layer_stride = row_stride * rows;
  const long long total = layer_stride * layers;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + (uintptr_t)total && d0 < s0 + (uintptr_t)total) return LS_ERR_INVALID_ARG;  // overlap
  if (!aligned(parent, 4)) return LS_ERR_INVALID_ARG;
  const Debug dbg = read_debug();
  if (dbg.check_ptrs) {
    if (!device_reachable(src) || !device_reachable(dst) || !device_reachable(parent)) return LS_ERR_INVALID_ARG;
    if (workspace && !device_reachable(workspace)) return LS_ERR_INVALID_ARG;
  }
  const long long slab_bytes = (long long)len * head_dim * es;
  int unit = 16;
  while (unit > 1 && ((s0 % unit) || (d0 % unit) || (slab_bytes % unit) || (slab_stride % unit))) unit >>= 1;
  const long long slab_units = slab_bytes / unit;
  if (slab_units * heads >= (1ll << 30) || rows >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (!di) return cuda_fail(cudaErrorUnknown);
  const int occ = copy_occupancy(di, unit);
  if (occ < 1) return cuda_fail(cudaErrorUnknown);

  ReorderParams p;
  p.src = static_cast<const unsigned char*>(src);
  p.dst = static_cast<unsigned char*>(dst);
  p.parent = parent;
  p.status = workspace ? reinterpret_cast<uint32_t*>(workspace) : nullptr;
  p.slab_stride = slab_stride;
  p.row_stride = row_stride;
  p.layer_stride = layer_stride;
  p.rows = (int)rows;
  p.k = k;
  p.heads = heads;
  p.layers = layers;
  p.slab_units = (int)slab_units;
  make_divisor((uint32_t)slab_units, &p.div_units_magic, &p.div_units_shift);
  p.pairs = (long long)layers * rows;
  const long long grid_full = (long long)di->sms * occ;
  const long long grid = p.pairs < grid_full ? p.pairs : grid_full;
  cudaError_t e = launch_cache_reorder(p, unit, (int)grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

ls_status ls_cache_refresh_inplace(void* cache, ls_dtype dtype, const int32_t* parent, int layers, int batch, int k,
                                   int heads, int max_len, int len, int head_dim, void* workspace, void* stream) {
  const ls_status ci = inplace_check_args(cache, dtype, parent, layers, batch, k, heads, max_len, len, head_dim,
                                          workspace);
  if (ci != LS_OK) return ci;
  if (layers == 0 || batch == 0 || heads == 0 || len == 0 || head_dim == 0) return LS_OK;
  const Debug dbg = read_debug();
  const long long es = dtype_bytes(dtype);
  const long long slab_stride = (long long)max_len * head_dim * es;
  const long long row_stride = slab_stride * heads;
  const long long layer_stride = row_stride * batch * k;
  const long long slab_bytes = (long long)len * head_dim * es;
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(cache);
  int unit = 16;
  while (unit > 1 && ((c0 % unit) || (slab_bytes % unit) || (slab_stride % unit))) unit >>= 1;
  const long long units = (long long)layers * batch * heads;
  if (units >= (1ll << 40) || (long long)batch * k >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (!di) return cuda_fail(cudaErrorUnknown);
  InplaceParams p;
  p.cache = static_cast<unsigned char*>(cache);
  p.parent = parent;
  p.status = workspace ? reinterpret_cast<uint32_t*>(workspace) : nullptr;
  p.work = nullptr;
  p.spin_limit_ns = dbg.spin_ns;
  p.layer_stride = layer_stride;
  p.row_stride = row_stride;
  p.slab_stride = slab_stride;
  p.slab_bytes = slab_bytes;
  p.batch = batch;
  p.k = k;
  p.heads = heads;
  p.layers = layers;
  p.units = units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // short slabs (up to 2 KB: the first 16 decode steps at c5) and k <= 8: the word kernel (a
  // warp per item, a lane per word position), about 256 words per item.  Measured at c5
  // against the bulk-copy kernel, one launch: len 1-4 9-15 us against 18-19 us, len 8-10
  // 27-33 us against 40-45 us, len 11-16 40-49 us against 43-51 us, about even at len 18-26.
  // Without bulk copies (unaligned slabs) it serves every length.
  const long long slab_words = slab_bytes / unit;
  const bool words_fit = k <= kIpWordMaxK && (long long)heads * slab_words < (1ll << 31) &&
                         (long long)batch * k <= kIpTmaMaxParents;
  const bool tma_fit = unit == 16 && (long long)batch * k <= kIpTmaMaxParents;
  const bool words = words_fit && !(dbg.flags & (kFlagPlainInplace | kFlagTmaInplace)) &&
                     (slab_bytes <= 2048 || !tma_fit || (dbg.flags & kFlagWordInplace));
  if (words) {
    long long wh = (dbg.ipw > 0 ? dbg.ipw : 256) / slab_words;
    wh = wh < 1 ? 1 : (wh > heads ? heads : wh);
    p.slab_words = slab_words;
    p.word_heads = (int)wh;
    make_divisor((uint32_t)slab_words, &p.word_magic, &p.word_shift);
    p.word_items = (long long)layers * batch * ((heads + wh - 1) / wh);
    p.tile_bytes = 0;
    p.heads_per_item = 0;
    const int wocc = inplace_words_occupancy(di, unit, batch, k);
    if (wocc < 1) return cuda_fail(cudaErrorUnknown);
    const long long warps_full = (long long)di->sms * wocc * (kIpWordThreads / 32);
    const long long warps = p.word_items < warps_full ? p.word_items : warps_full;
    const long long grid = (warps + kIpWordThreads / 32 - 1) / (kIpWordThreads / 32);
    const cudaError_t e = launch_cache_inplace_words(p, unit, (int)grid, st);
    return e == cudaSuccess ? LS_OK : cuda_fail(e);
  }
  // bulk copies when every slab and tile is 16-byte aligned and the parents fit in shared memory
  const bool tma = unit == 16 && (long long)batch * k <= kIpTmaMaxParents && !(dbg.flags & kFlagPlainInplace);
  const int tma_stage = dbg.ipstage >= 4096 && dbg.ipstage <= 64 * 1024 && dbg.ipstage % 16 == 0 ? dbg.ipstage : kIpTmaStage;
  const int occ = tma ? inplace_tma_occupancy(di, tma_stage, batch, k) : inplace_occupancy(di, unit);
  if (occ < 1) return cuda_fail(cudaErrorUnknown);
  const long long stage = tma ? tma_stage : kIpStageBytes;
  p.stage_bytes = tma_stage;
  const long long tile = (stage / k) / unit * unit;  // every row's tile fits one staging buffer
  p.tile_bytes = (int)(tile < slab_bytes ? tile : slab_bytes);
  // short slabs: an item of the bulk-copy kernel is as many heads of a (layer, batch) as fit a
  // buffer for ceil(k / 2) needed parents -- about what a beam-search batch needs -- and the
  // kernel moves an item in steps that fit the parents its batch actually needs (c5 loop, one
  // launch timed alone: 82.5 us sized for 2 parents, 83.5 for 3, 90.5 for all 4, 86.5 for 1);
  // the staged CTA kernel stages all k
  const long long k_item = !tma ? k : (dbg.ipkeff > 0 && dbg.ipkeff <= k ? dbg.ipkeff : (k + 1) / 2);
  long long hg = slab_bytes <= tile ? stage / (k_item * slab_bytes) : 1;
  hg = hg < 1 ? 1 : (hg > heads ? heads : hg);
  p.heads_per_item = (int)hg;
  const long long items = tma ? (long long)layers * batch * ((heads + hg - 1) / hg) *
                                    ((slab_bytes + p.tile_bytes - 1) / p.tile_bytes)
                              : units;
  const long long grid_full = (long long)di->sms * occ;
  const long long grid = items < grid_full ? items : grid_full;
  // with a workspace, the bulk-copy kernel's CTAs take items from a counter in it
  if (tma && workspace && items < (1ll << 31) && !(dbg.flags & kFlagStaticItems))
    p.work = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) + kIpWorkOff);
  const cudaError_t e = tma ? launch_cache_inplace_tma(p, (int)grid, st) : launch_cache_inplace(p, unit, (int)grid, st);
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

size_t ls_sample_workspace_size(int rows, int top_k, int vocab) {
  if (rows < 0 || top_k < 1 || top_k > LS_MAX_K || vocab < top_k) return 0;
  if (vocab > (1 << 28) || (long long)rows * ws_layout_sample(rows, top_k, vocab).nc_max >= (1ll << 31)) return 0;
  return ws_layout_sample(rows, top_k, vocab).total;
}

ls_status ls_sample(const void* logits, ls_dtype logit_dtype, const float* bias, const float* u, int rows, int vocab,
                    int top_k, float top_p, int32_t* out_token, float* out_logprob, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (rows < 0 || top_k < 1 || top_k > LS_MAX_K || vocab < top_k || vocab > (1 << 28)) return LS_ERR_INVALID_ARG;
  if (!(top_p > 0.0f) || !(top_p <= 1.0f)) return LS_ERR_INVALID_ARG;
  if (!dtype_ok(logit_dtype)) return LS_ERR_INVALID_ARG;
  if (rows == 0) return LS_OK;
  if (!logits || !u || !out_token || !workspace) return LS_ERR_INVALID_ARG;
  const WsLayout wl = ws_layout_sample(rows, top_k, vocab);
  if (wl.total == 0 || workspace_bytes < wl.total) return LS_ERR_INVALID_ARG;
  if ((long long)rows * wl.nc_max >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  const int es = dtype_bytes(logit_dtype);
  if (!aligned(logits, es) || (bias && !aligned(bias, 4)) || !aligned(u, 4) || !aligned(out_token, 4) ||
      (out_logprob && !aligned(out_logprob, 4)) || !aligned(workspace, 256))
    return LS_ERR_INVALID_ARG;
  const Debug dbg = read_debug();
  if (dbg.check_ptrs) {
    const void* ptrs[] = {logits, bias, u, out_token, out_logprob, workspace};
    for (const void* q : ptrs)
      if (q && !device_reachable(q)) return LS_ERR_INVALID_ARG;
  }
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (!di) return cuda_fail(cudaErrorUnknown);
  const int dtype = (int)logit_dtype;
  // the one-kernel sampler (K3's traversal, kFuSampRows rows per CTA, two strips a row) when
  // top_k <= 8, the CTAs fill the GPU by themselves and a strip's block maxima fit in shared
  // memory; otherwise K1 then K5
  {
    const int fu_parts = (kFuThreads / 32) / kFuSampRows;
    const int fu_vpl = (dtype == LS_DTYPE_F32 || bias) ? 4 : 8;
    const long long fu_ns = ((15 + (long long)vocab * es + 15) / 16 + 32ll * fu_vpl - 1) / (32ll * fu_vpl);
    const long long ctas = ((long long)rows + kFuSampRows - 1) / kFuSampRows;
    const bool one = !(dbg.flags & kFlagNoFused) && top_k <= kFuMaxK &&
                     (fu_ns + fu_parts - 1) / fu_parts <= kFuMaxStages &&
                     ((dbg.flags & kFlagFused) || 2 * ctas >= di->sms);
    if (one) {
      if (!fused_configured(di)) return cuda_fail(cudaErrorUnknown);
      unsigned char* ws = static_cast<unsigned char*>(workspace);
      StepParams p = {};
      p.logits = logits;
      p.bias = bias;
      p.u = u;
      p.out_token = out_token;
      p.out_logprob = out_logprob;
      p.top_p = top_p;
      p.status = reinterpret_cast<uint32_t*>(ws + wl.status_off);
      p.rowstat = reinterpret_cast<RowStat*>(ws + wl.rowstat_off);
      p.bstat = reinterpret_cast<int32_t*>(ws + wl.bstat_off);
      p.batch = (int)ctas;
      p.k = top_k;
      p.vocab = vocab;
      p.rows = rows;
      p.nc = fu_parts;
      p.stages = (int)((fu_ns + fu_parts - 1) / fu_parts);
      p.flags = dbg.flags;
      p.spin_limit_ns = dbg.spin_ns;
      const cudaError_t e = launch_sample_fused(p, dtype, static_cast<cudaStream_t>(stream));
      return e == cudaSuccess ? LS_OK : cuda_fail(e);
    }
  }
  RowPlan plan;
  const ls_status ps = plan_rows(di, dbg, dtype, es, bias != nullptr, vocab, rows, wl, &plan);
  if (ps != LS_OK) return ps;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // K1 over the rows: one row per sequence, top_k elements kept per row, none finished
  StepParams p = {};
  p.logits = logits;
  p.bias = bias;
  p.status = reinterpret_cast<uint32_t*>(ws + wl.status_off);
  p.done = reinterpret_cast<uint32_t*>(ws + wl.done_off);
  p.rec = ws + wl.rec_off;
  p.slots = reinterpret_cast<CandSlot*>(ws + wl.slot_off);
  p.rowstat = reinterpret_cast<RowStat*>(ws + wl.rowstat_off);
  p.bstat = reinterpret_cast<int32_t*>(ws + wl.bstat_off);
  p.batch = rows;
  p.k = top_k;
  p.vocab = vocab;
  p.rows = rows;
  p.nc = plan.nc;
  make_divisor((uint32_t)plan.nc, &p.nc_magic, &p.nc_shift);
  p.groups = wl.groups;
  p.slot_cap = wl.slot_cap;
  p.rec_stride = wl.rec_stride;
  p.flags = dbg.flags;
  p.units = plan.units;
  p.spin_limit_ns = dbg.spin_ns;
  SampleParams q;
  q.rec = p.rec;
  q.slots = p.slots;
  q.logits = logits;
  q.bias = bias;
  q.u = u;
  q.out_token = out_token;
  q.out_logprob = out_logprob;
  q.rowstat = p.rowstat;
  q.bstat = p.bstat;
  q.rows = rows;
  q.vocab = vocab;
  q.k = top_k;
  q.nc = plan.nc;
  q.groups = wl.groups;
  q.slot_cap = wl.slot_cap;
  q.rec_stride = wl.rec_stride;
  q.flags = dbg.flags;
  q.top_p = top_p;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_beam_rows(p, dtype, plan.vpl, (int)plan.grid, st);
  if (e == cudaSuccess) e = launch_sample_select(q, dtype, st);
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

ls_status ls_backtrack(const int32_t* token_hist, const int32_t* parent_hist, int steps, int batch, int k,
                       int eos_id, int32_t* out_seq, int32_t* out_len, void* workspace, void* stream) {
  if (steps < 0 || batch < 0 || k < 1 || k > LS_MAX_K) return LS_ERR_INVALID_ARG;
  if (steps == 0 || batch == 0) return LS_OK;
  if (!token_hist || !parent_hist || !out_seq || !out_len) return LS_ERR_INVALID_ARG;
  if ((long long)steps * batch * k >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  if (!aligned(token_hist, 4) || !aligned(parent_hist, 4) || !aligned(out_seq, 4) || !aligned(out_len, 4))
    return LS_ERR_INVALID_ARG;
  if (workspace && !aligned(workspace, 256)) return LS_ERR_INVALID_ARG;
  const Debug dbg = read_debug();
  if (dbg.check_ptrs) {
    const void* ptrs[] = {token_hist, parent_hist, out_seq, out_len, workspace};
    for (const void* q : ptrs)
      if (q && !device_reachable(q)) return LS_ERR_INVALID_ARG;
  }
  BacktrackParams p;
  p.tok = token_hist;
  p.par = parent_hist;
  p.seq = out_seq;
  p.len = out_len;
  p.status = workspace ? reinterpret_cast<uint32_t*>(workspace) : nullptr;
  p.steps = steps;
  p.batch = batch;
  p.k = k;
  p.eos = eos_id;
  p.tile = backtrack_tile(k, steps);
  const cudaError_t e = launch_backtrack(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

ls_status ls_read_status(void* workspace, void* stream) {
  if (!workspace) return LS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof word, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (word & kDevTimeout) return LS_ERR_TIMEOUT;
  if (word & (kDevBadParent | kDevInternal)) return LS_ERR_INTERNAL;
  return LS_OK;
}

const char* ls_status_string(ls_status status) {
  switch (status) {
    case LS_OK: return "ok";
    case LS_ERR_INVALID_ARG: return "invalid argument";
    case LS_ERR_UNSUPPORTED: return "unsupported request";
    case LS_ERR_CUDA: return "CUDA runtime error";
    case LS_ERR_TIMEOUT: return "bounded device wait timed out";
    case LS_ERR_INTERNAL: return "device-detected internal error (e.g. parent index out of range)";
    default: return "unknown status";
  }
}

ls_status ls_read_row_stats(const void* workspace, int batch, int k, int vocab, float* lse, float* rtopk,
                            int32_t* ncand, int32_t* path, void* stream) {
  if (!workspace || batch < 0 || k < 1 || k > LS_MAX_K || vocab < k) return LS_ERR_INVALID_ARG;
  if (batch == 0) return LS_OK;
  const WsLayout wl = ws_layout(batch, k, vocab);
  const size_t rows = (size_t)batch * k;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned char* ws = static_cast<const unsigned char*>(workspace);
  RowStat* tmp = static_cast<RowStat*>(std::malloc(rows * sizeof(RowStat)));
  int32_t* bs = static_cast<int32_t*>(std::malloc((size_t)batch * sizeof(int32_t)));
  if (!tmp || !bs) {
    std::free(tmp);
    std::free(bs);
    return LS_ERR_INTERNAL;
  }
  cudaError_t e = cudaMemcpyAsync(tmp, ws + wl.rowstat_off, rows * sizeof(RowStat), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(bs, ws + wl.bstat_off, (size_t)batch * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) {
    for (size_t r = 0; r < rows; ++r) {
      if (lse) lse[r] = tmp[r].lse;
      if (rtopk) rtopk[r] = tmp[r].rtopk;
      if (ncand) ncand[r] = tmp[r].ncand;
    }
    if (path) std::memcpy(path, bs, (size_t)batch * sizeof(int32_t));
  }
  std::free(tmp);
  std::free(bs);
  return e == cudaSuccess ? LS_OK : cuda_fail(e);
}

}  // extern "C"
