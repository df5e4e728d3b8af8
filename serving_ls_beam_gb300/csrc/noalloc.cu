// ls_beam_step_noalloc: the beam step for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocating routine: code that runs inside
// a host framework which owns every byte of device memory and forbids allocations from
// its plugins, and serving loops with a fixed memory budget where an allocation at
// request time could stall or fail.  For them the scratch space of the beam step lives
// in one fixed-size array in this library's own device memory, reserved when the
// library's device code is loaded and held on every GPU that loads it until the
// process exits.  The caller still passes inputs and outputs.
//
// Limits and sharing: shapes whose scratch (ls_beam_step_workspace_size) exceeds
// kNoAllocScratchBytes are rejected.  Every call uses the same array and leaves its
// contents behind; the status word (device-detected errors, e.g. a bounded wait that ran
// out) is cleared at the start of each call and read with ls_beam_step_noalloc_status
// before the next one.  Calls whose work overlaps on the GPU (different streams, or
// different host threads without ordering) race on the array and must not be issued.
// The array's device address is looked up once per device; a cudaDeviceReset unloads the
// library's device code with the context, so the library is not used on a device after
// one.
#include <cuda_runtime.h>

#include <mutex>

#include "ls_beam.h"
#include "ls_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up once per device,
// with that device current).  In host code the array's name is only a host-side stand-in,
// so kernels must be given this address, never the name.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" ls_status ls_beam_step_noalloc(const void* logits, ls_dtype logit_dtype, const float* bias,
                                          const float* beam_scores, const uint8_t* finished, int batch, int k,
                                          int vocab, int eos_id, int32_t* out_token, int32_t* out_parent,
                                          float* out_score, uint8_t* out_finished, void* stream) {
  // every argument check of ls_beam_step first: a rejected call touches nothing on the GPU
  const ls_status chk = lsb::beam_step_check_args(logits, logit_dtype, bias, beam_scores, finished, batch, k,
                                                  vocab, eos_id, out_token, out_parent, out_score, out_finished);
  if (chk != LS_OK || batch == 0) return chk;
  const size_t need = ls_beam_step_workspace_size(batch, k, vocab);
  if (need == 0) return LS_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return LS_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = scratch_address();
  if (!scratch) return LS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word must start at zero; everything else the step reads it writes first
  if (cudaMemsetAsync(scratch, 0, 256, st) != cudaSuccess) {
    cudaGetLastError();
    return LS_ERR_CUDA;
  }
  return ls_beam_step(logits, logit_dtype, bias, beam_scores, finished, batch, k, vocab, eos_id, out_token,
                      out_parent, out_score, out_finished, scratch, kNoAllocScratchBytes, stream);
}

extern "C" ls_status ls_beam_step_noalloc_status(void* stream) {
  void* scratch = scratch_address();
  if (!scratch) return LS_ERR_CUDA;
  return ls_read_status(scratch, stream);  // the status word is the array's first word
}
