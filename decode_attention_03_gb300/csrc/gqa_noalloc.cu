// gqa_decode_noalloc: the contiguous decode step for callers that cannot hand the
// library a device workspace -- for example a plugin whose device memory is
// budgeted and owned by a host framework, a latency-critical loop in which
// cudaMalloc's implicit synchronisation is not acceptable, or a plain C / FFI
// caller that has no device allocator at all.
//
// The split partials and arrival counters live in one file-scope device array of
// GQA_NOALLOC_SCRATCH_BYTES per GPU (held by every GPU that loads the library,
// until the process exits).  Nothing here allocates: no cudaMalloc, no cudaFree,
// no allocating library routine.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gqa_decode.h"
#include "gqa_kernels.cuh"   // the status word's bits (kDevTimeout, kDevBadInput)

static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kStatusBytes = 4;   // the device status word at the start of the array
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in; the real address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
gqa_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return GQA_ERR_CUDA;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return GQA_OK;
}

}  // namespace

extern "C" gqa_status gqa_decode_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                                         int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head,
                                         float scale, void* stream) {
  const size_t need = gqa_decode_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head, 0);
  if (need == 0) {
    // invalid shape (or no usable device): let the regular entry point name the error
    return gqa_decode(q, k, v, o, batch, T_q, S_kv, h_q, h_kv, d_head, scale, nullptr, 0, stream);
  }
  if (need > GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_WORKSPACE;
  if (batch == 0) return GQA_OK;
  void* scratch = nullptr;
  gqa_status s = scratch_on_current_device(&scratch);
  if (s != GQA_OK) return s;
  // the arrival counters must start at zero, and the array keeps the previous call's contents:
  // clear everything the header and counters span except the status word, which keeps the
  // error bits of earlier calls until gqa_decode_noalloc_check reads them.  Split partials need
  // no clearing: a call that completes without a device fault writes every partial it reads
  // (after a fault the outputs are invalid anyway, and the check reports it).
  const size_t zeroed = gqa_decode_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head, 1);
  if (zeroed <= kStatusBytes || zeroed > GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_INVALID_ARG;
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + kStatusBytes, 0, zeroed - kStatusBytes,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GQA_ERR_CUDA;
  return gqa_decode(q, k, v, o, batch, T_q, S_kv, h_q, h_kv, d_head, scale, scratch, GQA_NOALLOC_SCRATCH_BYTES,
                    stream);
}

extern "C" gqa_status gqa_decode_noalloc_check(void* stream) {
  void* scratch = nullptr;
  gqa_status s = scratch_on_current_device(&scratch);
  if (s != GQA_OK) return s;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GQA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GQA_ERR_CUDA;
  if (word != 0 && cudaMemset(scratch, 0, sizeof(word)) != cudaSuccess) return GQA_ERR_CUDA;
  if (word & gqa::kDevBounds) return GQA_ERR_BOUNDS;
  if (word & gqa::kDevTimeout) return GQA_ERR_TIMEOUT;
  if (word & gqa::kDevBadInput) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}
