// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/lora_sgmv.h"

namespace lsg {

// Bound of every wait inside a kernel (build-time knob; a test build shortens it).
#ifndef LSG_WAIT_LIMIT_NS
#define LSG_WAIT_LIMIT_NS 2000000000ull
#endif

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int round_up(int a, int b) { return ceil_div(a, b) * b; }

// ---- segmentation
struct SegPlan {
  int nw;             // warps (each owns one histogram row and one chunk of tokens)
  bool gmem;          // histograms in the workspace instead of shared memory
  size_t ws_bytes;    // workspace bytes required
  size_t smem_bytes;  // dynamic shared memory bytes
};
SegPlan seg_plan(int n, int P);
lora_status launch_segment(const int32_t* ids, int n, int P, int32_t* perm, int32_t* seg_offsets,
                           int32_t* seg_adapter, int32_t* num_segments, int32_t* hist, int32_t* err_flag,
                           cudaStream_t stream);

// ---- SGMV (CUDA-core split-K path)
constexpr int kMaxProj = LORA_MAX_PROJ;

struct ProjArgs {
  const uint16_t* x;
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* y;
  int64_t ldx, ldy;
  int32_t h_in, h_out;
  float scale;
};

enum Mode : int { kModeShrink = 1, kModeExpand = 2, kModeFused = 3 };

struct SgmvCall {
  Mode mode;
  ProjArgs proj[kMaxProj];
  int n_proj;
  int r;
  int n_adapters;
  lora_segments seg;
  float* v_out;       // shrink output [n][r]
  // Shrink mode: v_out may hold up to v_parts_max slices [n][r]; the
  // tensor-tile kernel then splits each long tile's k-blocks into that many
  // parts at most, slice p holding the partial sum of part p (the sum over
  // the slices is v).  The number of slices written goes to *v_parts
  // (host memory) when v_parts is not null.  0 or 1: v_out is v itself.
  int32_t v_parts_max;
  int32_t* v_parts;
  const float* v_in;  // expand input [n][r]
  int32_t* err_flag;
  // Slot arenas (null slot_of: each pool is contiguous, [n_adapters] slabs of
  // rank r).  Adapter a lives in slot slot_of[a] with rank rank_of[a], a bit
  // of rank_mask (bit c: rank 8 << c); a slot holds rank <= r_max.
  const int32_t* slot_of;
  const int32_t* rank_of;
  int n_slots;
  int r_max;
  unsigned rank_mask;
  // One-launch step: the adapter ids of the batch; the call segments them
  // into seg's buffers itself (inside the SGMV launch when the batch is small,
  // else with lora_segment first, using seg_hist as its workspace).
  const int32_t* ids;
  int32_t* seg_hist;
  // (sgmv_multi_host) the ids in host memory: they travel in the launch's
  // parameters when the batch is segmented inside the launch (ids above is
  // then not written), else they are copied to ids first
  const int32_t* ids_host;
  // The long segments were handled by another launch (the backbone GEMM with
  // the fused expand): this call skips them and launches no tensor-tile kernel.
  int32_t long_done;
};

lora_status launch_sgmv_cc(const SgmvCall& call, cudaStream_t stream);

// ---- SGMV (tcgen05 tile path for long segments)
// Segments of at least kLongSeg tokens go to the tensor-tile kernel when it
// applies (a batch where segments can be long; every mode and rank); the
// split-K kernel skips exactly those segments then.
constexpr int kLongSeg = 64;
bool sgmv_tc_applicable(const SgmvCall& call);
lora_status launch_sgmv_tc(const SgmvCall& call, cudaStream_t stream);

// ---- backbone GEMM with the LoRA expand fused into its epilogue
constexpr int kGlVParts = 4;  // k-partial slices of v the shrink may write
struct GemmLoraCall {
  const uint16_t* x;
  int64_t ldx;
  const uint16_t* W;  // [h_in][h_out]
  const uint16_t* A_pool;
  const uint16_t* B_pool;
  int32_t n_adapters, h_in, h_out, r;
  float scale;
  lora_segments seg;
  uint16_t* y;
  int64_t ldy;
  float* v;  // workspace [kGlVParts][n][r]: the shrink's k-partial slices
  int32_t* err_flag;
};
lora_status launch_gemm_lora(const GemmLoraCall& call, cudaStream_t stream);

// TMA tensor map over bf16 data: `rank` dims (innermost first), byte strides
// of dims 1.., box extents in elements, swizzle span in bytes (0 = none).
lora_status encode_tmap_bf16(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
                             const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes);

// Records a CUDA error from a runtime call; returns LORA_ERR_CUDA on failure.
lora_status cuda_status(cudaError_t e);

#ifdef LSG_TEST_HOOKS
// Test builds only: the kernels withhold one signal (1: the decode kernel's
// end-of-work marker, 2: the partial v that CTA 1 of each decode cluster
// pushes, 3: the tensor-tile kernel's first expand accumulator, 4: the
// backbone GEMM's first completed accumulator pair), so a bounded wait runs
// out; 0: none.
lora_status test_withhold_cc(int what);
lora_status test_withhold_tc(int what);
lora_status test_withhold_gl(int what);
#endif

}  // namespace lsg
