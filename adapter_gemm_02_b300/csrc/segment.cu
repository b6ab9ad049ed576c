// lora_segment: group a batch's tokens by adapter.
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary),
// "Interesting ideas" I2: sort the batch by adapter so that same-adapter
// requests sit next to each other and form dense segments; "Summary":
// requests of the same adapter are grouped.
//
// One CTA runs a stable counting sort (batches of more than 256 tokens; smaller
// ones take the rank sort below, which needs no histogram over the pool).  Warp w owns the w-th contiguous chunk
// of tokens and one histogram row H[w][0..P] (bucket P collects invalid ids,
// so they land after every valid token).  Steps: per-warp counts (warp-match
// aggregated, no atomics: the row is private to the warp), per-key exclusive
// scan over warps, block-wide exclusive scan over keys (giving segment starts)
// fused with the compaction of the non-empty adapters, then a stable scatter
// where each warp walks its chunk in order and ranks equal keys inside a
// 32-token group by warp match.  Rows live in shared memory unless the pool is
// too large, in which case they live in the caller's workspace.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace lsg {

constexpr size_t kSegSmemBudget = 200 * 1024;
constexpr int kSegScratchInts = 128;  // block-scan partials, in shared memory

constexpr int kSegRankTokens = 256;  // batches up to this size take the rank sort (no histogram)

SegPlan seg_plan(int n, int P) {
  SegPlan pl{};
  if (n >= 1 && n <= kSegRankTokens) {  // the rank sort's batches (an empty batch takes the counting sort)
    pl.nw = 1;
    pl.gmem = false;
    pl.ws_bytes = 0;
    pl.smem_bytes = 0;
    return pl;
  }
  const int want = std::clamp(std::max(ceil_div(std::max(n, 1), 64), ceil_div(P + 1, 256)), 1, 32);
  const size_t row = static_cast<size_t>(P + 1) * sizeof(int32_t);
  const size_t scratch = kSegScratchInts * sizeof(int32_t);
  auto need = [&](int w) { return static_cast<size_t>(w + 1) * row + scratch; };
  pl.nw = want;
  if (need(1) <= kSegSmemBudget) {
    while (pl.nw > 1 && need(pl.nw) > kSegSmemBudget) pl.nw /= 2;
    pl.gmem = false;
    pl.ws_bytes = 0;
    pl.smem_bytes = need(pl.nw);
  } else {
    pl.gmem = true;
    pl.ws_bytes = static_cast<size_t>(pl.nw + 1) * row;
    pl.smem_bytes = scratch;
  }
  return pl;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

__global__ void __launch_bounds__(1024)
    lora_segment_kernel(const int32_t* __restrict__ ids, int n, int P, int max_segments,
                        int32_t* __restrict__ perm, int32_t* __restrict__ seg_offsets,
                        int32_t* __restrict__ seg_adapter, int32_t* __restrict__ num_segments,
                        int32_t* gbuf, int32_t* err_flag) {
  extern __shared__ __align__(16) int32_t sbuf[];
  // The SGMV launch that follows may start its prologue now; it reads our
  // outputs only after griddepcontrol.wait, i.e. after this grid completes.
  pdl_launch_dependents();
  // Our own inputs (ids) and outputs may be in use by the previous launch.
  pdl_wait();

  const int nt = blockDim.x, nw = nt >> 5, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Pp = P + 1;
  int32_t* H = gbuf ? gbuf : sbuf;                    // [nw][Pp]
  int32_t* TOT = H + static_cast<size_t>(nw) * Pp;    // [Pp]
  int32_t* scratch = gbuf ? sbuf : (TOT + Pp);        // kSegScratchInts

  const size_t hsize = static_cast<size_t>(nw) * Pp;
  for (size_t i = tid; i < hsize; i += nt) H[i] = 0;
  __syncthreads();

  // 1. per-warp histogram of its chunk
  const int chunk = (n + nw - 1) / nw;
  const int lo = min(n, warp * chunk), hi = min(n, lo + chunk);
  int32_t* Hw = H + static_cast<size_t>(warp) * Pp;
  bool bad_seen = false;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool act = i < hi;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int a = ids[i];
      const int key = (a >= 0 && a < P) ? a : P;
      bad_seen |= (key == P);
      const unsigned peers = __match_any_sync(am, key);
      if (lane == __ffs(peers) - 1) Hw[key] += __popc(peers);
    }
    __syncwarp();
  }
  if (bad_seen) set_err(err_flag, LORA_ERR_BAD_ADAPTER_ID);
  __syncthreads();

  // 2. per key: exclusive scan across warps, column total into TOT
  for (int a = tid; a < Pp; a += nt) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const size_t idx = static_cast<size_t>(w) * Pp + a;
      const int c = H[idx];
      H[idx] = run;
      run += c;
    }
    TOT[a] = run;
  }
  __syncthreads();

  // 3. block exclusive scan over keys of (count, non-empty flag); writes the
  //    segment start of every key and compacts non-empty adapters.
  const int per = (Pp + nt - 1) / nt;
  const int a0 = min(Pp, tid * per), a1 = min(Pp, a0 + per);
  int sum = 0, cnt = 0;
  for (int a = a0; a < a1; ++a) {
    const int c = TOT[a];
    sum += c;
    cnt += (a < P && c > 0);
  }
  const int xs = warp_incl_scan(sum, lane), xc = warp_incl_scan(cnt, lane);
  if (lane == 31) {
    scratch[warp] = xs;
    scratch[32 + warp] = xc;
  }
  __syncthreads();
  if (warp == 0) {
    const int s = lane < nw ? scratch[lane] : 0;
    const int c = lane < nw ? scratch[32 + lane] : 0;
    const int is = warp_incl_scan(s, lane), ic = warp_incl_scan(c, lane);
    __syncwarp();
    scratch[lane] = is - s;
    scratch[32 + lane] = ic - c;
    if (lane == 31) {
      scratch[64] = is;
      scratch[65] = ic;
    }
  }
  __syncthreads();
  int run_s = scratch[warp] + xs - sum;
  int run_c = scratch[32 + warp] + xc - cnt;
  for (int a = a0; a < a1; ++a) {
    const int c = TOT[a];
    TOT[a] = run_s;
    if (a < P && c > 0) {
      seg_adapter[run_c] = a;
      seg_offsets[run_c] = run_s;
      ++run_c;
    }
    run_s += c;
  }
  __syncthreads();
  const int S = scratch[65];
  const int n_valid = TOT[P];
  if (tid == 0) *num_segments = S;
  for (int s = S + tid; s <= max_segments; s += nt) seg_offsets[s] = n_valid;
  for (int s = S + tid; s < max_segments; s += nt) seg_adapter[s] = -1;

  // 4. cursors: first output slot of (warp, key)
  for (size_t i = tid; i < hsize; i += nt) H[i] += TOT[i % Pp];
  __syncthreads();

  // 5. stable scatter: warps walk their chunks in token order
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool act = i < hi;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int a = ids[i];
      const int key = (a >= 0 && a < P) ? a : P;
      const unsigned peers = __match_any_sync(am, key);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int b = Hw[key];
      perm[b + rank] = i;
      __syncwarp(am);
      if (lane == __ffs(peers) - 1) Hw[key] = b + __popc(peers);
    }
    __syncwarp();
  }
}

// The same segmentation for a small batch (n <= kSegRankMaxTokens), one thread
// per token and no histogram over the pool.  Token i's place in the stable
// order is the number of tokens that sort before it: a smaller id, or the
// same id at a smaller index (tokens j < i count when id_j <= id_i, tokens
// j > i when id_j < id_i), counted over all ids in shared memory.  The sorted
// ids then mark the segments: sorted position t starts one when its id is
// valid and differs from position t - 1's, and its segment index is the
// number of such starts before it (a block-wide prefix count).  Ids outside
// [0, P) sort as P, after every valid id, in no segment.
constexpr int kSegRankMaxTokens = kSegRankTokens;

__global__ void __launch_bounds__(kSegRankMaxTokens)
    lora_segment_rank_kernel(const int32_t* __restrict__ ids, int n, int P, int max_segments,
                             int32_t* __restrict__ perm, int32_t* __restrict__ seg_offsets,
                             int32_t* __restrict__ seg_adapter, int32_t* __restrict__ num_segments,
                             int32_t* err_flag) {
  __shared__ __align__(16) int32_t keys[kSegRankMaxTokens];
  __shared__ int32_t skeys[kSegRankMaxTokens];
  __shared__ int32_t warp_starts[kSegRankMaxTokens / 32];
  pdl_launch_dependents();
  pdl_wait();
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5, nw = blockDim.x >> 5;
  constexpr int kPad = 0x7fffffff;  // threads past n: after every token
  int key = kPad;
  bool bad = false;
  if (i < n) {
    const int id = ids[i];
    bad = id < 0 || id >= P;
    key = bad ? P : id;
  }
  keys[i] = key;
  __syncthreads();
  // place in the stable order (blockDim is a multiple of 32: whole int4 groups)
  const int4* k4 = reinterpret_cast<const int4*>(keys);
  const int i4 = i >> 2, n4 = blockDim.x >> 2;
  int pos = 0;
  for (int j4 = 0; j4 < i4; ++j4) {
    const int4 v = k4[j4];
    pos += (v.x <= key) + (v.y <= key) + (v.z <= key) + (v.w <= key);
  }
  {
    const int4 v = k4[i4];
    const int e = i & 3;  // the group holding token i: j < i counts <=, j > i counts <
    pos += (e > 0 ? v.x <= key : v.x < key) + (e > 1 ? v.y <= key : (e < 1 && v.y < key)) +
           (e > 2 ? v.z <= key : (e < 2 && v.z < key)) + (e < 3 && v.w < key);
  }
  for (int j4 = i4 + 1; j4 < n4; ++j4) {
    const int4 v = k4[j4];
    pos += (v.x < key) + (v.y < key) + (v.z < key) + (v.w < key);
  }
  if (i < n) {
    perm[pos] = i;
    skeys[pos] = key;
  }
  if (bad) set_err(err_flag, LORA_ERR_BAD_ADAPTER_ID);
  __syncthreads();
  // sorted position t = i: a segment starts here when the id is valid and new
  const int sk = i < n ? skeys[i] : kPad;
  const bool valid = sk < P;
  const bool start = valid && (i == 0 || skeys[i - 1] != sk);
  const unsigned sb = __ballot_sync(0xffffffffu, start);
  if (lane == 0) warp_starts[warp] = __popc(sb);
  const int n_valid = __syncthreads_count(valid);
  int seg = __popc(sb & ((1u << lane) - 1u));
  int S = 0;
  for (int w = 0; w < nw; ++w) {
    const int c = warp_starts[w];
    seg += w < warp ? c : 0;
    S += c;
  }
  if (start) {
    seg_adapter[seg] = sk;
    seg_offsets[seg] = i;
  }
  for (int x = S + i; x <= max_segments; x += blockDim.x) seg_offsets[x] = n_valid;
  for (int x = S + i; x < max_segments; x += blockDim.x) seg_adapter[x] = -1;
  if (i == 0) *num_segments = S;
}

lora_status launch_segment(const int32_t* ids, int n, int P, int32_t* perm, int32_t* seg_offsets,
                           int32_t* seg_adapter, int32_t* num_segments, int32_t* hist, int32_t* err_flag,
                           cudaStream_t stream) {
  if (n >= 1 && n <= kSegRankMaxTokens) {
    // small batch: the rank sort (needs no workspace whatever the pool)
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[1];
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(static_cast<unsigned>(round_up(n, 32)));
    cfg.stream = stream;
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, lora_segment_rank_kernel, ids, n, P, std::min(n, P), perm,
                                          seg_offsets, seg_adapter, num_segments, err_flag));
  }
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  cudaError_t attr_err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(lora_segment_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSegSmemBudget));
  });
  if (attr_err != cudaSuccess) return LORA_ERR_CUDA;
  const SegPlan pl = seg_plan(n, P);
  // the counting sort's rows (nw + 1 of P + 1 ints) and scan scratch must fit the
  // shared memory it is given (rows in the workspace: the scratch alone)
  const size_t rows_bytes = static_cast<size_t>(pl.nw + 1) * (static_cast<size_t>(P) + 1) * sizeof(int32_t);
  const size_t need = (pl.gmem ? 0 : rows_bytes) + kSegScratchInts * sizeof(int32_t);
  if (pl.smem_bytes < need || (pl.gmem && hist == nullptr)) return LORA_ERR_UNSUPPORTED;
  const int max_segments = std::min(n, P);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[1];
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(pl.nw * 32);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = stream;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int32_t* gbuf = pl.gmem ? hist : nullptr;
  return cuda_status(cudaLaunchKernelEx(&cfg, lora_segment_kernel, ids, n, P, max_segments, perm, seg_offsets,
                                        seg_adapter, num_segments, gbuf, err_flag));
}

}  // namespace lsg
