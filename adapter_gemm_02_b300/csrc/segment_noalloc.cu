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
// array's name as a device address, so its address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made in a
// CUDA context; the address is cached per context (by the driver's unique
// context id), so a context created later (after cudaDeviceReset, or one made
// current through the driver API) looks it up again instead of reusing an
// address that belonged to a destroyed or foreign context.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace lsg {
namespace {

constexpr size_t kNoAllocScratchBytes = LORA_SEGMENT_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) int32_t g_segment_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

struct ScratchEntry {
  unsigned long long ctx_id;  // 0: unused (the driver's context ids start at 1)
  int32_t* ptr;
};
constexpr int kEntries = 64;
std::mutex g_mu;
ScratchEntry g_cache[kEntries] = {};
int g_next = 0;

PFN_cuCtxGetCurrent_v4000 g_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_get_id = nullptr;
std::once_flag g_once;

// Unique id of the CUDA context current on this thread (after the runtime has
// made the device's primary context current if none was).
lora_status current_context_id(unsigned long long* id) {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (g_get_current == nullptr || g_get_id == nullptr) return LORA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_get_current(&ctx) != CUDA_SUCCESS) return LORA_ERR_CUDA;
  if (ctx == nullptr) {
    // no context current on this thread yet: make the device's primary context current
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return LORA_ERR_CUDA;
    if (g_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return LORA_ERR_CUDA;
  }
  if (g_get_id(ctx, id) != CUDA_SUCCESS || *id == 0) return LORA_ERR_CUDA;
  return LORA_OK;
}

// Device address of g_segment_scratch in the current context (looked up on
// the first call in each context).
lora_status scratch_in_current_context(int32_t** out) {
  unsigned long long id = 0;
  if (const lora_status s = current_context_id(&id); s != LORA_OK) return s;
  std::lock_guard<std::mutex> lk(g_mu);
  for (const ScratchEntry& e : g_cache)
    if (e.ctx_id == id) {
      *out = e.ptr;
      return LORA_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_segment_scratch) != cudaSuccess || p == nullptr) return LORA_ERR_CUDA;
  g_cache[g_next] = ScratchEntry{id, static_cast<int32_t*>(p)};
  g_next = (g_next + 1) % kEntries;
  *out = static_cast<int32_t*>(p);
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
    const lora_status s = scratch_in_current_context(&scratch);
    if (s != LORA_OK) return s;
  }
  return launch_segment(ids, n_tokens, n_adapters, perm, seg_offsets, seg_adapter, num_segments, scratch,
                        err_flag, reinterpret_cast<cudaStream_t>(stream));
}
