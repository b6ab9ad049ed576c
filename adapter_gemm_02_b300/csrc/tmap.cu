// Host-side encoding of TMA tensor maps through the driver entry point
// cuTensorMapEncodeTiled (looked up once through the runtime, so the library
// does not link libcuda directly).  Encoding costs tens of microseconds of
// host time, so encoded maps are kept in a small per-thread cache keyed by
// every encoding argument (the adapter pools of a model are the same buffers
// call after call).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "internal.h"

namespace lsg {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

}  // namespace

namespace {

struct TmapKey {
  const void* base;
  int32_t rank, swizzle;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
};

struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool used;
};

constexpr int kCacheEntries = 64;
thread_local TmapEntry t_cache[kCacheEntries];
thread_local int t_next = 0;

TmapKey make_key(const void* base, int rank, const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                 int swizzle) {
  TmapKey k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.rank = rank;
  k.swizzle = swizzle;
  for (int i = 0; i < rank && i < 3; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  return k;
}

}  // namespace

lora_status encode_tmap_bf16(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
                             const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
  if (rank < 1 || rank > 3) return LORA_ERR_INVALID_ARG;
  const TmapKey key = make_key(base, rank, dims, strides_bytes, box, swizzle_bytes);
  for (int i = 0; i < kCacheEntries; ++i) {
    if (t_cache[i].used && std::memcmp(&t_cache[i].key, &key, sizeof(key)) == 0) {
      *out = t_cache[i].map;
      return LORA_OK;
    }
  }
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode == nullptr) return LORA_ERR_CUDA;
  cuuint64_t gdim[5];
  cuuint64_t gstr[4];
  cuuint32_t bdim[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) gstr[i] = strides_bytes[i];
  }
  CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
  if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUresult r = g_encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                              const_cast<void*>(base), gdim, gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return LORA_ERR_CUDA;
  TmapEntry& e = t_cache[t_next];
  t_next = (t_next + 1) % kCacheEntries;
  e.key = key;
  e.map = *out;
  e.used = true;
  return LORA_OK;
}

}  // namespace lsg
