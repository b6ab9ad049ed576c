// Adapter loading into slot arenas: copies into a slot and table entries.
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Summary":
// adapters are loaded on demand, in milliseconds.  A slot of capacity r_max
// holds one adapter's A as [h_in][rank] and B as [rank][h_out], packed at the
// slot start, so each matrix is one contiguous copy; the table entry that
// names the slot is written afterwards on the same stream, so a batch
// ordered after it sees the whole adapter.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace lsg {
namespace {

__global__ void slot_assign_kernel(int32_t* slot_of, int32_t* rank_of, int32_t adapter, int32_t slot,
                                   int32_t rank) {
  if (threadIdx.x == 0) {
    slot_of[adapter] = slot;
    rank_of[adapter] = rank;
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool is_rank(int r) { return r == 8 || r == 16 || r == 32 || r == 64; }

}  // namespace
}  // namespace lsg

using namespace lsg;

extern "C" {

lora_status lora_slot_copy(const lora_slot_src* srcs, int32_t n_src, int32_t n_slots, int32_t r_max, int32_t slot,
                           int32_t rank, lora_stream_t stream) {
  if (!srcs || n_src < 1 || n_slots < 1) return LORA_ERR_INVALID_ARG;
  if (slot < 0 || slot >= n_slots) return LORA_ERR_INVALID_ARG;
  if (!is_rank(r_max) || !is_rank(rank) || rank > r_max) return LORA_ERR_UNSUPPORTED;
  for (int i = 0; i < n_src; ++i) {
    const lora_slot_src& s = srcs[i];
    if (!s.A_arena || !s.B_arena || !s.A_src || !s.B_src) return LORA_ERR_INVALID_ARG;
    if (s.h_in < 8 || s.h_out < 8 || (s.h_in % 8) || (s.h_out % 8)) return LORA_ERR_UNSUPPORTED;
    if (!al16(s.A_arena) || !al16(s.B_arena)) return LORA_ERR_MISALIGNED;
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  for (int i = 0; i < n_src; ++i) {
    const lora_slot_src& s = srcs[i];
    const size_t a_elems = static_cast<size_t>(s.h_in) * rank, b_elems = static_cast<size_t>(rank) * s.h_out;
    lora_bf16* a_dst = s.A_arena + static_cast<size_t>(slot) * s.h_in * r_max;
    lora_bf16* b_dst = s.B_arena + static_cast<size_t>(slot) * r_max * s.h_out;
    if (cudaMemcpyAsync(a_dst, s.A_src, a_elems * 2, cudaMemcpyDefault, st) != cudaSuccess) return LORA_ERR_CUDA;
    if (cudaMemcpyAsync(b_dst, s.B_src, b_elems * 2, cudaMemcpyDefault, st) != cudaSuccess) return LORA_ERR_CUDA;
  }
  return LORA_OK;
}

lora_status lora_slot_assign(int32_t* slot_of, int32_t* rank_of, int32_t n_adapters, int32_t adapter, int32_t slot,
                             int32_t rank, lora_stream_t stream) {
  if (!slot_of || !rank_of || n_adapters < 1) return LORA_ERR_INVALID_ARG;
  if (!al4(slot_of) || !al4(rank_of)) return LORA_ERR_MISALIGNED;
  if (adapter < 0 || adapter >= n_adapters || slot < -1) return LORA_ERR_INVALID_ARG;
  if (slot >= 0 && !is_rank(rank)) return LORA_ERR_UNSUPPORTED;
  slot_assign_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(slot_of, rank_of, adapter, slot,
                                                                           slot >= 0 ? rank : 0);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
