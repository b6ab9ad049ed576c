// lora_segment_noalloc: lora_segment for callers that cannot allocate device
// memory, e.g. code that runs while its framework owns the allocator, inside
// a real-time loop whose memory was planned up front, or in a plugin given
// only its input and output buffers.  lora_segment needs a caller-provided
// workspace once the adapter pool is too large for its per-warp histograms to
// fit in shared memory; this variant takes that scratch from a fixed-size
// array in device global memory that the library owns instead.
//
// The array is file-scope device memory: every GPU that loads the library
// holds it until the process exits.  All calls share it (it keeps whatever the
// last call left; the kernel clears the part it uses on entry), so two calls
// whose kernels overlap on the GPU race on it.  Host code cannot use the
// array's name as a device address, so the address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace lsg {
namespace {

constexpr size_t kNoAllocScratchBytes = LORA_SEGMENT_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) int32_t g_segment_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_segment_scratch on the current device (looked up once).
lora_status scratch_on_current_device(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LORA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_segment_scratch) != cudaSuccess || p == nullptr) return LORA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return LORA_OK;
}

}  // namespace
}  // namespace lsg

using namespace lsg;

extern "C" lora_status lora_segment_noalloc(const int32_t* ids, int32_t n_tokens, int32_t n_adapters,
                                            int32_t* perm, int32_t* seg_offsets, int32_t* seg_adapter,
                                            int32_t* num_segments, int32_t* err_flag, lora_stream_t stream) {
  if (n_tokens < 0 || n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (!seg_offsets || !num_segments) return LORA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!ids || !perm || !seg_adapter)) return LORA_ERR_INVALID_ARG;
  const SegPlan pl = seg_plan(n_tokens, n_adapters);
  int32_t* scratch = nullptr;
  if (pl.gmem) {
    if (pl.ws_bytes > kNoAllocScratchBytes) return LORA_ERR_WORKSPACE;
    const lora_status s = scratch_on_current_device(&scratch);
    if (s != LORA_OK) return s;
  }
  return launch_segment(ids, n_tokens, n_adapters, perm, seg_offsets, seg_adapter, num_segments, scratch,
                        err_flag, reinterpret_cast<cudaStream_t>(stream));
}
