// SGMV for short segments (decode), the HBM-bound regime.
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Summary":
// the per-adapter low-rank additions of a mixed batch are computed together,
// requests of one adapter grouped into segments; "Key points": SGMV runs on
// the GPU's tensor cores, and rank is far below the hidden size (16 vs 4096).
// For a decode segment the work is a few rank-r dot products per token, so
// time goes to streaming the adapter's A and B slabs from HBM; this kernel is
// built to keep HBM busy with as few instructions per byte as possible:
//
//  * Work item = (token tile of <= T tokens of one segment, projection).  A
//    cluster of C CTAs takes one item: CTA `rank` streams rows
//    [rank*k_chunk, +k_chunk) of A (split-K of the shrink) and columns
//    [rank*n_chunk, +n_chunk) of B (split-N of the expand).
//  * One producer warp fills a shared-memory ring of 2-3 stages of 24-28 KiB
//    (mbarrier transaction counts) with 2-D TMA tensor copies of the A rows
//    (swizzled to the row width, so the fragment loads below are free of bank
//    conflicts) and of the B block [r][columns], and with one bulk copy per
//    token for the gathered x / y row pieces.  It runs ahead across items, so
//    the next item's slabs stream while the current item is reduced.
//  * Four consumer warps run warp-level tensor-core MMAs (m16n8k16, bf16 in,
//    fp32 accumulate) with the tile's tokens as the M rows: the shrink splits
//    the stage's k-steps over the warps, the warps' partial v are summed in
//    shared memory, and each CTA pushes its partial v into every peer's shared
//    memory with st.async (completing as transaction bytes on the peer's
//    mbarrier) and sums the C partials in a fixed order, so every CTA holds
//    the identical fp32 v, which never leaves the chip in the fused mode.  The
//    expand takes v as a pair of bf16 MMA operands (v = hi + lo, hi = bf16(v),
//    lo = bf16(v - hi); the pair carries 16 bits of v's mantissa), adds
//    s * v.B to y in fp32 and stores y rounded once to bf16.
//  * Persistent grid: as many clusters as are co-resident; cluster g takes
//    items g, g+G, ... in tile-major order (all projections of a tile in a
//    row), read from the device-side segmentation without a host round trip.
//
// Partial-v buffers are double-buffered by item parity and need no extra
// synchronisation: a peer can push item j+2 only after it received our
// partial of item j+1, which we send after we finished reading item j.
//
// Modes: shrink (v -> device memory), expand (v from device memory, no
// cluster), fused (v on chip).
//
// Adapter pools: a contiguous pool ([n_adapters][h_in][r], one rank) or slot
// arenas (fixed-size slots of capacity r_max, adapter a in slot slot_of[a]
// with rank rank_of[a], its A packed as [h_in][rank] and its B as
// [rank][h_out] at the slot start).  A kernel compiled for a set of ranks
// takes each item's rank from the table and runs the rank's code (fragment
// counts, swizzle, stage shape) for that item; the ring is shaped for the
// largest rank of the set.  Ranks stay far below the hidden size and
// adapters of different ranks share a batch ([Punica-el] "Key points").
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "seg_warp.cuh"

namespace lsg {

// Ring shape per rank (build-time knobs, chosen by measurement on B300):
// two stages, 16 KiB at r = 8, 24 KiB at r = 16 and 28 KiB at r = 32, so that
// one CTA's share of a decode item (A rows + B columns + x/y pieces) is in
// flight at once and three to four CTAs share an SM (larger r = 8 / 16 stages
// and 32 or 40 KiB at r = 32 measured slower); r = 64, whose CTAs registers
// hold to two per SM, keeps three 28 KiB stages in flight.
#ifndef LSG_CC_STAGES_SMALL
#define LSG_CC_STAGES_SMALL 2
#endif
#ifndef LSG_CC_KB_SMALL
#define LSG_CC_KB_SMALL 24
#endif
#ifndef LSG_CC_STAGES_BIG
#define LSG_CC_STAGES_BIG 3
#endif
#ifndef LSG_CC_STAGES_R8
#define LSG_CC_STAGES_R8 LSG_CC_STAGES_SMALL
#endif
#ifndef LSG_CC_KB_BIG
#define LSG_CC_KB_BIG 28
#endif
#ifndef LSG_CC_KB_R8
#define LSG_CC_KB_R8 16
#endif
#ifndef LSG_CC_STAGES_R32
#define LSG_CC_STAGES_R32 LSG_CC_STAGES_SMALL
#endif
#ifndef LSG_CC_KB_R32
#define LSG_CC_KB_R32 28
#endif
// Tiles of 4 tokens when segments hold at most this many tokens on average
// (the tokens per possible segment), else of 16.
#ifndef LSG_CC_T4_MAX_AVG
#define LSG_CC_T4_MAX_AVG 3.0
#endif
#ifndef LSG_CC_WARPS
#define LSG_CC_WARPS 4
#endif
#ifndef LSG_CC_ROWS_PER_CTA
#define LSG_CC_ROWS_PER_CTA 512
#endif
constexpr int kCW = LSG_CC_WARPS;      // consumer warps
constexpr int kCThreads = kCW * 32;    // consumer threads
constexpr int kThreads = kCThreads + 32;
constexpr int kMaxC = 8;               // CTAs per cluster (portable limit)
constexpr int kXB = 2;                 // partial-v exchange buffers
// 1: a one-launch step's ids (up to 64) are loaded at the kernel's entry
#ifndef LSG_CC_IDS_EARLY
#define LSG_CC_IDS_EARLY 1
#endif
constexpr uint64_t kWaitLimitNs = LSG_WAIT_LIMIT_NS;  // per wait (2 s)

#ifdef LSG_TEST_HOOKS
__device__ int g_test_withhold;
__device__ __forceinline__ bool withhold(int what) { return *(volatile int*)&g_test_withhold == what; }
lora_status test_withhold_cc(int what) { return cuda_status(cudaMemcpyToSymbol(g_test_withhold, &what, sizeof(int))); }
#else
__device__ __forceinline__ bool withhold(int) { return false; }
#endif

enum : int { kStShrink = 1, kStExpand = 2, kStFirst = 4, kStLast = 8, kStEnd = 16 };

// A set of ranks as bits: 8 -> 1, 16 -> 2, 32 -> 4, 64 -> 8.
constexpr int kAllRanks = 15;
__host__ __device__ constexpr int rank_bit(int r) { return r == 8 ? 1 : r == 16 ? 2 : r == 32 ? 4 : r == 64 ? 8 : 0; }
__host__ __device__ constexpr int rank_class(int r) { return r == 8 ? 0 : r == 16 ? 1 : r == 32 ? 2 : 3; }
__host__ __device__ constexpr int set_max_rank(int set) { return (set & 8) ? 64 : (set & 4) ? 32 : (set & 2) ? 16 : 8; }
__host__ __device__ constexpr bool single_rank(int set) { return set == 1 || set == 2 || set == 4 || set == 8; }

// Runs f(integral_constant<int, r>) for the rank r of the set (a single-rank
// set needs no test).
template <int RSET, class F>
__device__ __forceinline__ void with_rank(int r, F&& f) {
  if constexpr (single_rank(RSET)) {
    f(std::integral_constant<int, set_max_rank(RSET)>{});
  } else {
    if constexpr ((RSET & 1) != 0)
      if (r == 8) return f(std::integral_constant<int, 8>{});
    if constexpr ((RSET & 2) != 0)
      if (r == 16) return f(std::integral_constant<int, 16>{});
    if constexpr ((RSET & 4) != 0)
      if (r == 32) return f(std::integral_constant<int, 32>{});
    if constexpr ((RSET & 8) != 0)
      if (r == 64) return f(std::integral_constant<int, 64>{});
  }
}

struct CCProj {
  const uint16_t* x;
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* y;
  int64_t ldx, ldy;
  int32_t h_in, h_out;
  int32_t k_chunk, n_chunk;  // rows of A / columns of B per rank (k_chunk: multiple of 16)
  float scale;
};

// Everything but the tensor maps; copied to shared memory at kernel start so
// that no later access waits on a constant-cache miss.
struct CCTail {
  CCProj proj[kMaxProj];
  const int32_t* perm;
  const int32_t* seg_offsets;
  const int32_t* seg_adapter;
  const int32_t* num_segments;
  float* v_out;
  const float* v_in;
  int32_t* err_flag;
  int32_t n_proj;
  int32_t n_tokens;
  int32_t max_segments;
  int32_t n_adapters;
  int32_t csplit;     // C
  int32_t skip_long;  // segments of >= kLongSeg tokens belong to the tensor-tile kernel
  int32_t tc_ranks;   // slot arenas: ranks (rank_bit) whose long segments the tensor-tile kernel took
  const int32_t* slot_of;  // slot of each adapter (null: adapter a lives in slot a)
  const int32_t* rank_of;  // rank of each adapter (null: every adapter has the kernel's rank)
  int32_t n_slots;
  int32_t rmax;                    // slot capacity in ranks (the contiguous pool: its rank)
  int32_t rank_mask;               // ranks that have tensor maps in this launch (rank_bit)
  int32_t map_of[kMaxProj][4];     // tensor-map pair of (projection, rank class), -1: none
  int32_t map_bw[kMaxProj];        // B box width of a map pair (columns, an odd multiple of 8)
  int32_t map_nb[kMaxProj];        // B boxes per expand stage of a map pair
  // One-launch step: the producer warp of every CTA segments ids itself (in
  // the shared memory past CCSmem) and CTA 0 writes the segmentation to
  // perm / seg_offsets / seg_adapter / num_segments.  Null: segmentation given.
  const int32_t* ids;
};

// Map pair m serves one (projection, rank r): tmA views the projection's A
// storage as 2-D rows of r elements ([n_slots*h_in*rmax/r][r], box {r, BA}:
// slot s starts at row s*h_in*rmax/r), tmB views its B storage as
// [n_slots*rmax][h_out] (box {bw, r}: slot s starts at row s*rmax).
// ids of a one-launch step that come from host memory travel in the
// parameters (read by the producer warp from the constant bank)
constexpr int kIdsInParamsMax = 128;
struct CCParams {
  CUtensorMap tmA[kMaxProj];
  CUtensorMap tmB[kMaxProj];
  CCTail t;
  int32_t n_ids_in_params;  // > 0: the one-launch step's ids are ids_in_params[0 .. n)
  int32_t ids_in_params[kIdsInParamsMax];
};

// Rank R's stage contents in a ring shaped for rank RM >= R.
template <int R, int T, int RM = R>
struct CCCfg {
  static constexpr int kStages = RM >= 64   ? LSG_CC_STAGES_BIG
                                : RM == 8  ? LSG_CC_STAGES_R8
                                : RM == 32 ? LSG_CC_STAGES_R32
                                           : LSG_CC_STAGES_SMALL;
  static constexpr int kStageBytes =
      (RM >= 64 ? LSG_CC_KB_BIG : RM == 8 ? LSG_CC_KB_R8 : RM == 32 ? LSG_CC_KB_R32 : LSG_CC_KB_SMALL) * 1024;
  // shrink: A rows per stage (A part + x part fit a stage), whole k-steps of
  // 16, made of NBA TMA boxes of BA rows (a box extent is at most 256)
  static constexpr int WS0 = (((kStageBytes - T * 16) / ((R + T) * 2)) / 16) * 16;
  static constexpr int NBA = (WS0 + 255) / 256;
  static constexpr int BA = ((WS0 / NBA) / 16) * 16;
  static constexpr int WS = NBA * BA;
  static constexpr int XP = WS + 8;              // x / y row pitch: an odd number of 16-byte chunks
  static constexpr int kPartBytes = WS * R * 2;  // x / y part starts here
  static constexpr int SWA = R >= 16 ? R * 2 : 0;  // A-part swizzle span in bytes (0: none)
  static constexpr uint32_t SWM = SWA ? SWA / 16 - 1 : 0;
  static constexpr int NT = R / 8;               // 8-rank n-tiles of the shrink
  static constexpr int KS = R / 16;              // 16-rank k-steps of the expand (0 for r = 8)
  static_assert(WS >= 16 && BA >= 16, "stage too small");
  static_assert(kPartBytes + T * XP * 2 <= kStageBytes, "stage overflow");
  static_assert(T * R % 4 == 0, "exchange layout");
  static_assert(T <= 16, "one MMA row block");
};

template <int T>
struct StageHdr {
  int32_t kind;
  int32_t proj;
  int32_t tlen;
  int32_t len;    // rows (shrink) or columns (expand) in this stage
  int32_t off;    // first row / column
  int32_t pitch;  // expand: box width (columns) of the B part
  int32_t rk;     // the item's rank
  int32_t tok[T];
};

// Shared memory of a kernel whose largest rank is R (smaller ranks use the
// leading part of red / xbuf / vfull, as [.][T][r] arrays).
template <int R, int T>
struct CCSmem {
  static constexpr int kStages = CCCfg<R, T>::kStages;
  alignas(1024) uint8_t ring[kStages][CCCfg<R, T>::kStageBytes];
  alignas(16) CCTail t;
  StageHdr<T> hdr[kStages];
  alignas(8) uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t xbar[kXB];
  alignas(16) float red[kCW][T][R];
  alignas(16) float xbuf[kXB][kMaxC][T][R];
  alignas(16) float vfull[T][R];
  alignas(16) uint16_t zero_row[8];  // fragment rows past the tile's tokens read this
  int32_t abort;                     // a consumer warp gave up on a wait: every warp stops
};

// Barrier of the consumer warps.  Returns false once a consumer warp has given
// up on a wait (the abort flag): the caller then leaves its loop.
__device__ __forceinline__ bool consumer_sync(const int32_t* abort) {
  named_bar_sync(1, kCThreads);
  return *reinterpret_cast<const volatile int32_t*>(abort) == 0;
}

__device__ __forceinline__ uint32_t ld_shared_u32(const void* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// bf16x2 {lo: a, hi: b} from two floats (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Cursor over the segments, 32 at a time (one per lane), finding token tile
// `tile` (tiles of <= T tokens, segment by segment).  Tile indices a CTA asks
// for only grow.  The first window is loaded together with num_segments, so
// locating the first tile costs one round trip.  Executed by a full warp.
template <int T>
struct SegCursor {
  int base = 0, tiles_before = 0, S = 0;
  int off = 0, len = 0, ad = -1;  // segment base + lane
  int sl = -1, rk = 0;            // its adapter's slot and rank (0: the kernel's rank)

  __device__ void load(const CCTail& q, int lane, int bound) {
    const int s = base + lane;
    off = 0;
    len = 0;
    ad = -1;
    sl = -1;
    rk = 0;
    if (s < bound) {
      const int o = q.seg_offsets[s];
      const int e = q.seg_offsets[s + 1];
      ad = q.seg_adapter[s];
      off = o;
      len = (o >= 0 && e <= q.n_tokens && e >= o) ? e - o : 0;
      sl = ad;
      if (q.slot_of != nullptr && ad >= 0 && ad < q.n_adapters) {
        sl = q.slot_of[ad];
        rk = q.rank_of[ad];
      }
      if (q.skip_long && len >= kLongSeg) {
        // taken by the tensor-tile kernel (with slot arenas: valid slot, a rank it ran)
        const bool tc_took = q.slot_of == nullptr || (sl >= 0 && sl < q.n_slots && (rank_bit(rk) & q.tc_ranks));
        if (tc_took) len = 0;
      }
    }
  }

  __device__ void init(const CCTail& q, int lane) {
    const int s_raw = *q.num_segments;
    load(q, lane, min(32, q.max_segments));  // speculative: issued alongside num_segments
    S = min(max(s_raw, 0), q.max_segments);
    if (lane >= S) len = 0;
  }

  __device__ bool find(const CCTail& q, int lane, int tile, int& t0, int& tlen, int& a, int& slot, int& r) {
    while (base < S) {
      const int tl = (len + T - 1) / T;
      int inc = tl;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
      }
      const int total = __shfl_sync(0xffffffffu, inc, 31);
      if (tile < tiles_before + total) {
        const unsigned m = __ballot_sync(0xffffffffu, tiles_before + inc > tile);
        const int ls = __ffs(m) - 1;
        const int excl = __shfl_sync(0xffffffffu, inc - tl, ls);
        const int o = __shfl_sync(0xffffffffu, off, ls);
        const int l = __shfl_sync(0xffffffffu, len, ls);
        a = __shfl_sync(0xffffffffu, ad, ls);
        slot = __shfl_sync(0xffffffffu, sl, ls);
        r = __shfl_sync(0xffffffffu, rk, ls);
        t0 = o + (tile - tiles_before - excl) * T;
        tlen = min(T, o + l - t0);
        return true;
      }
      tiles_before += total;
      base += 32;
      load(q, lane, S);
    }
    return false;
  }
};

// RSET: the ranks this kernel runs (a single rank for a contiguous pool or a
// one-rank slot table; several for a slot table of mixed ranks).
template <int RSET, int T, int MODE>
__global__ void __launch_bounds__(kThreads) sgmv_cc_kernel(const __grid_constant__ CCParams p) {
  constexpr int RM = set_max_rank(RSET);
  using CfgM = CCCfg<RM, T>;
  constexpr int kStages = CfgM::kStages;
  constexpr bool kHasShrink = (MODE & kModeShrink) != 0;
  constexpr bool kHasExpand = (MODE & kModeExpand) != 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  auto& sm = *reinterpret_cast<CCSmem<RM, T>*>(smem_raw);
  const CCTail& q = sm.t;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = p.t.csplit;
  const int rank = static_cast<int>(blockIdx.x) % C;
  const int group = static_cast<int>(blockIdx.x) / C;
  const int ngroups = static_cast<int>(gridDim.x) / C;
  const bool xchg = kHasShrink && C > 1;

  // One-launch step of up to 64 tokens: the producer's lanes load the ids
  // first, so that their latency overlaps the prologue below (the ids are
  // read before the dependency wait, as the header states).
  int id_pre[2] = {0, 0};
  auto load_ids = [&]() {
    const int32_t* ids = p.n_ids_in_params > 0 ? p.ids_in_params : p.t.ids;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = e * 32 + lane;
      if (i < p.t.n_tokens) id_pre[e] = ids[i];
    }
  };
  if (LSG_CC_IDS_EARLY && warp == kCW && p.t.ids != nullptr && p.t.n_tokens <= 64) load_ids();

  // Per-call parameters to shared memory: every word in flight at once.
  {
    static_assert(sizeof(CCTail) % 4 == 0, "tail size");
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&p.t);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.t);
    for (int i = tid; i < static_cast<int>(sizeof(CCTail) / 4); i += kThreads) dst[i] = src[i];
  }
  if (warp == kCW && lane < kMaxProj) {
    if (kHasShrink) prefetch_tmap(&p.tmA[lane]);
    if (kHasExpand) prefetch_tmap(&p.tmB[lane]);
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
    }
    for (int b = 0; b < kXB; ++b) mbar_init(&sm.xbar[b], 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (tid < 8) sm.zero_row[tid] = 0;
  __syncthreads();
  // Our mbarriers exist before any peer pushes into this CTA: every thread
  // arrives now and waits before its first push (or at the end).
  if (xchg) cluster_arrive_relaxed();
  // The next launch may begin its prologue; it waits for our completion before
  // touching memory.  Before reading x, y, v or a segmentation record, and
  // before writing anything, we wait for the preceding launch in the stream
  // (which may write them).  The producer warp reads the token ids and the
  // adapter pools first: those are never written by the launch it overlaps.
  pdl_launch_dependents();
  if (warp != kCW) pdl_wait();
  // The swizzle below is computed on absolute shared addresses, which agrees
  // with the TMA's when the ring starts on a 1 KiB boundary (all CTAs alike).
  const bool ring_ok = (smem_u32(sm.ring) & 1023u) == 0;

  if (warp == kCW) {
    // ============================== producer warp
    int slot = 0;
    uint32_t phase = 0;
    bool failed = !ring_ok;
    if (!ring_ok && lane == 0) set_err(q.err_flag, LORA_ERR_UNSUPPORTED);
    // the preceding launch in the stream has completed (waited for once, just
    // before this warp first reads x / y or a given segmentation record; then
    // CTA 0 writes the segmentation it computed to the caller's buffers)
    bool dep = false;
    WarpSegOut so{0, 0, false};
    auto wait_dep = [&]() {
      if (dep) return;
      pdl_wait();
      dep = true;
      if (q.ids != nullptr && blockIdx.x == 0) {
        // the caller's segmentation buffers, as lora_segment fills them
        const int n = q.n_tokens, ms = q.max_segments;
        int32_t* perm_g = const_cast<int32_t*>(p.t.perm);
        int32_t* offs_g = const_cast<int32_t*>(p.t.seg_offsets);
        int32_t* adap_g = const_cast<int32_t*>(p.t.seg_adapter);
        for (int i = lane; i < n; i += 32) perm_g[i] = q.perm[i];
        for (int x = lane; x <= ms; x += 32) offs_g[x] = x <= so.S ? q.seg_offsets[x] : so.n_valid;
        for (int x = lane; x < ms; x += 32) adap_g[x] = x < so.S ? q.seg_adapter[x] : -1;
        if (lane == 0) *const_cast<int32_t*>(p.t.num_segments) = so.S;
        if (__any_sync(0xffffffffu, so.bad) && lane == 0) set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
      }
      __syncwarp();
    };
    if (q.ids != nullptr) {
      const int n = q.n_tokens, P = q.n_adapters, ms = q.max_segments;
      // the sort's temporaries (ids, key cursors) in ring stage 0, which no
      // copy has touched yet; the result past CCSmem, kept for the cursor
      int32_t* ids_s = reinterpret_cast<int32_t*>(sm.ring[0]);
      int32_t* cnt = ids_s + n;
      int32_t* perm_s = reinterpret_cast<int32_t*>(smem_raw + sizeof(CCSmem<RM, T>));
      int32_t* offs_s = perm_s + n;
      int32_t* adap_s = offs_s + ms + 1;
      int32_t* count_s = adap_s + max(ms, 1);
      // up to 64 tokens: ranks in registers; more: counting sort in shared memory
      const int32_t* ids = p.n_ids_in_params > 0 ? p.ids_in_params : q.ids;
      if (!LSG_CC_IDS_EARLY && n <= 64) load_ids();
      so = n <= 32   ? warp_segment_rank<1>(id_pre, n, P, perm_s, offs_s, adap_s, lane)
           : n <= 64 ? warp_segment_rank<2>(id_pre, n, P, perm_s, offs_s, adap_s, lane)
                     : warp_segment(ids, n, P, ids_s, cnt, perm_s, offs_s, adap_s, lane);
      fence_proxy_async_smem();  // stage 0 is next written by the tensor copies
      if (lane == 0) *count_s = so.S;
      __syncwarp();
      // the cursor reads the shared-memory copy
      if (lane == 0) {
        sm.t.perm = perm_s;
        sm.t.seg_offsets = offs_s;
        sm.t.seg_adapter = adap_s;
        sm.t.num_segments = count_s;
      }
      __syncwarp();
    }
    // a given segmentation record (and a slot table) may come from the preceding launch
    if (q.ids == nullptr) wait_dep();
    SegCursor<T> cur;
    cur.init(q, lane);
    int last_tile = -1, a = -1, sl = -1, rk = 0, t0 = 0, tlen = 0, tok = -1, ntok = 0, tk = -1;
    bool tile_ok = false, tok_ready = false;

    // stages this warp has filled (bit s) and the phase parity of each one's
    // last fill: drained before the CTA leaves after a failed wait
    uint32_t filled = 0, fill_par = 0;
    auto acquire = [&]() -> bool {
      bool ok = *reinterpret_cast<volatile int32_t*>(&sm.abort) == 0;
      if (ok && lane == 0) ok = mbar_wait(&sm.empty[slot], phase ^ 1u, kWaitLimitNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && lane == 0) set_err(q.err_flag, LORA_ERR_TIMEOUT);
      return ok;
    };
    auto advance = [&]() {
      filled |= 1u << slot;
      fill_par = (fill_par & ~(1u << slot)) | (phase << slot);
      if (++slot == kStages) {
        slot = 0;
        phase ^= 1u;
      }
    };
    // validate the tile's token indices (loaded when the tile was found)
    auto resolve_tok = [&]() {
      tok = tk;
      if (lane < tlen && (tok < 0 || tok >= q.n_tokens)) {
        set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
        tok = -1;
      }
      ntok = __popc(__ballot_sync(0xffffffffu, tok >= 0));
      tok_ready = true;
    };
    auto header = [&](int kind, int pj, int len, int off, int pitch) {
      StageHdr<T>& h = sm.hdr[slot];
      if (lane < T) h.tok[lane] = tok;
      if (lane == 0) {
        h.kind = kind;
        h.proj = pj;
        h.tlen = tlen;
        h.len = len;
        h.off = off;
        h.pitch = pitch;
        h.rk = rk;
      }
      __syncwarp();
    };

    for (int item = group; !failed; item += ngroups) {
      const int tile = item / q.n_proj;
      const int pj = item - tile * q.n_proj;
      if (tile != last_tile) {
        if (!cur.find(q, lane, tile, t0, tlen, a, sl, rk)) break;
        last_tile = tile;
        tk = -1;
        if (lane < tlen) tk = q.perm[t0 + lane];  // consumed after the first A copy is issued
        tok_ready = false;
        if (rk == 0) rk = RM;
        // a rank outside the launch's mask has no tensor map: the item is skipped
        tile_ok = a >= 0 && a < q.n_adapters && sl >= 0 && sl < q.n_slots &&
                  (rank_bit(rk) & RSET & q.rank_mask) != 0 && rk <= q.rmax;
        if (!tile_ok && lane == 0) set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
      }
      if (!tile_ok) continue;  // every CTA of the cluster skips it alike
      const CCProj& pr = q.proj[pj];

      with_rank<RSET>(rk, [&](auto rc) {
        constexpr int R = decltype(rc)::value;
        using Cfg = CCCfg<R, T, RM>;
        const int mi = q.map_of[pj][rank_class(R)];
        if (kHasShrink) {
          const int k0 = rank * pr.k_chunk;
          const int klen = max(0, min(pr.h_in, k0 + pr.k_chunk) - k0);
          const int nst = max(1, (klen + Cfg::WS - 1) / Cfg::WS);
          const int per = ((klen + nst - 1) / nst + 15) & ~15;
          const int arow = sl * pr.h_in * (q.rmax / R);  // first row of the adapter's A in the map
          for (int st = 0; st < nst; ++st) {
            const int r0 = k0 + st * per;
            const int rl = max(0, min(per, k0 + klen - r0));
            const int nbx = (rl + Cfg::BA - 1) / Cfg::BA;  // A boxes in this stage
            if (!acquire()) {
              failed = true;
              break;
            }
            uint8_t* st_base = sm.ring[slot];
            if (lane == 0 && nbx) mbar_expect_tx(&sm.full[slot], static_cast<uint32_t>(nbx) * Cfg::BA * R * 2u);
            if (lane < nbx)
              tma_load_2d(st_base + lane * Cfg::BA * R * 2, &p.tmA[mi], 0, arow + r0 + lane * Cfg::BA,
                          &sm.full[slot]);
            wait_dep();  // x rows next
            if (!tok_ready) resolve_tok();
            header(kStShrink | (st == 0 ? kStFirst : 0) | (st == nst - 1 ? kStLast : 0), pj, rl, r0, 0);
            if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], static_cast<uint32_t>(rl) * 2u * ntok);
            if (rl > 0 && tok >= 0)
              bulk_g2s(st_base + Cfg::kPartBytes + lane * Cfg::XP * 2,
                       pr.x + static_cast<int64_t>(tok) * pr.ldx + r0, rl * 2, &sm.full[slot]);
            advance();
          }
        }
        if (kHasExpand && !failed) {
          const int c0 = rank * pr.n_chunk;
          const int clen = max(0, min(pr.h_out, c0 + pr.n_chunk) - c0);
          const int bw = q.map_bw[mi];
          const int sc = bw * q.map_nb[mi];  // columns per stage
          const int nst = (clen + sc - 1) / sc;
          const int brow = sl * q.rmax;  // first row of the adapter's B in the map
          wait_dep();  // y rows next
          if (!tok_ready) resolve_tok();
          for (int st = 0; st < nst; ++st) {
            const int cc = c0 + st * sc;
            const int cl = min(sc, c0 + clen - cc);
            const int nbs = (cl + bw - 1) / bw;  // boxes in this stage
            if (!acquire()) {
              failed = true;
              break;
            }
            uint8_t* st_base = sm.ring[slot];
            if (lane == 0) mbar_expect_tx(&sm.full[slot], static_cast<uint32_t>(nbs) * bw * R * 2u);
            if (lane < nbs)
              tma_load_2d(st_base + lane * bw * R * 2, &p.tmB[mi], cc + lane * bw, brow, &sm.full[slot]);
            header(kStExpand | (st == 0 ? kStFirst : 0) | (st == nst - 1 ? kStLast : 0), pj, cl, cc, bw);
            if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], static_cast<uint32_t>(cl) * 2u * ntok);
            if (tok >= 0)
              bulk_g2s(st_base + Cfg::kPartBytes + lane * Cfg::XP * 2,
                       pr.y + static_cast<int64_t>(tok) * pr.ldy + cc, cl * 2, &sm.full[slot]);
            advance();
          }
        }
      });
    }
    wait_dep();  // also when this CTA had no item: CTA 0 writes the segmentation
    if (!failed && acquire()) {
      if (lane == 0 && !withhold(1)) {
        sm.hdr[slot].kind = kStEnd;
        mbar_arrive(&sm.full[slot]);
      }
    } else if (!ring_ok) {
      // nothing was issued: tell the consumers to stop
      if (lane == 0) {
        sm.hdr[0].kind = kStEnd;
        mbar_arrive(&sm.full[0]);
      }
    } else if (lane == 0) {
      // a wait failed: no copy issued by this warp may still be landing in
      // shared memory when the CTA leaves (bounded waits for each stage's
      // last fill; a stage the consumers already took completes at once)
      for (int s2 = 0; s2 < kStages; ++s2)
        if (filled & (1u << s2)) (void)mbar_wait(&sm.full[s2], (fill_par >> s2) & 1u, kWaitLimitNs);
    }
    if (xchg) {
      cluster_wait_acquire();   // start barrier
      cluster_arrive_relaxed();  // end barrier: no CTA leaves while a peer may still push to it
      cluster_wait_acquire();
    }
    return;
  }

  // ============================== consumer warps
  const int ct = tid;  // 0 .. kCThreads-1
  const int g = lane >> 2, tig = lane & 3;  // MMA fragment coordinates
  const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix lm, row lr of it
  int slot = 0;
  uint32_t phase = 0;
  int nx = 0;  // partial-v exchanges done
  bool start_waited = false;
  // (sized for the largest rank; a smaller rank uses the leading entries)
  float acc[CfgM::NT][4];  // this warp's partial v: rows g, g+8 of every 8-rank n-tile
  // expand operands: v as bf16 hi/lo MMA A fragments (per 16-rank k-step)
  constexpr int KSA = CfgM::KS > 0 ? CfgM::KS : 1;
  uint32_t vah[KSA][4], val[KSA][4];
  uint32_t v8h[2] = {0u, 0u}, v8l[2] = {0u, 0u};  // r = 8: one m16n8k8 A fragment
#pragma unroll
  for (int ks = 0; ks < KSA; ++ks)
#pragma unroll
    for (int e = 0; e < 4; ++e) vah[ks][e] = val[ks][e] = 0u;
#pragma unroll
  for (int n = 0; n < CfgM::NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
  bool quit = false;
  int xarm = -1;  // exchange buffer armed for the current item's peer partials, until they are in
  // This warp gives up on a wait: the error, the abort flag, and one arrival
  // at the consumer barrier, which releases warps that wait there (or will)
  // so that they read the flag and leave as well.
  auto give_up = [&]() {
    if (lane == 0) {
      set_err(q.err_flag, LORA_ERR_TIMEOUT);
      *reinterpret_cast<volatile int32_t*>(&sm.abort) = 1;
    }
    __threadfence_block();
    __syncwarp();
    named_bar_arrive(1, kCThreads);
    quit = true;
  };

  for (;;) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&sm.full[slot], phase, kWaitLimitNs);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      give_up();
      break;
    }
    const StageHdr<T>& h = sm.hdr[slot];
    const int kind = h.kind;
    if (kind & kStEnd) break;
    const int tlen = h.tlen, len = h.len, off = h.off, pj = h.proj;
    const uint8_t* st_base = sm.ring[slot];

    with_rank<RSET>(h.rk, [&](auto rc) {
      constexpr int R = decltype(rc)::value;
      using Cfg = CCCfg<R, T, RM>;
      constexpr int NT = Cfg::NT;
      // this rank's views of the exchange buffers
      auto& red = *reinterpret_cast<float(*)[kCW][T][R]>(&sm.red[0][0][0]);
      auto& xbuf = *reinterpret_cast<float(*)[kXB][kMaxC][T][R]>(&sm.xbuf[0][0][0][0]);
      auto& vfull = *reinterpret_cast<float(*)[T][R]>(&sm.vfull[0][0]);
      if (kind & kStShrink) {
        const int b = nx & 1;
        if (kind & kStFirst) {
  #pragma unroll
          for (int n = 0; n < NT; ++n)
  #pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
          if (xchg && ct == 0)
            mbar_arrive_expect_tx(&sm.xbar[b], static_cast<uint32_t>(C - 1) * T * R * 4u);
          if (xchg) xarm = b;
        }
        // ---- v[t, :] += x[t, k-range] . A[k-range, :]  (tokens = MMA rows)
        const uint32_t a_base = smem_u32(st_base);
        const uint32_t x_base = a_base + Cfg::kPartBytes;
        const int nk16 = len >> 4;
        // x fragment (A operand): lane L gives row (L/8 & 1)*8 + L%8, k offset (L/16)*8 of the
        // 16x16 block; rows past the tile read the zero row
        const int xrow = (lm & 1) * 8 + lr;
        const uint32_t xaddr0 = xrow < tlen ? x_base + static_cast<uint32_t>(xrow * Cfg::XP + (lm >> 1) * 8) * 2
                                            : smem_u32(sm.zero_row);
        const uint32_t xstep = xrow < tlen ? 32u : 0u;  // bytes per k-step of 16
        // A fragment (B operand, swizzled rows of R ranks): per-lane offset, independent of the k-step
        const int krow = (lm & 1) * 8 + lr;
        auto step = [&](int ks, auto& ac) {  // ac: float[>= NT][4]
          uint32_t a0, a1, a2, a3;
          ldsm_x4(xaddr0 + static_cast<uint32_t>(ks) * xstep, a0, a1, a2, a3);
          const uint32_t kbase = a_base + static_cast<uint32_t>(ks) * (16 * R * 2);
          if constexpr (NT == 1) {
            // r = 8: matrices (k 0-7), (k 8-15) of the single n-tile; lanes 16+ repeat 0-15
            uint32_t b0, b1;
            ldsm_x2_trans(kbase + static_cast<uint32_t>(krow) * (R * 2), b0, b1);
            mma_bf16_16816(ac[0], a0, a1, a2, a3, b0, b1);
          } else {
  #pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              // matrices: (k 0-7, n 0-7), (k 8-15, n 0-7), (k 0-7, n 8-15), (k 8-15, n 8-15) of the pair
              const uint32_t off = swz<Cfg::SWM>(static_cast<uint32_t>(krow) * (R * 2) +
                                                 static_cast<uint32_t>(np * 16 + (lm >> 1) * 8) * 2);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_trans(kbase + off, b0, b1, b2, b3);
              mma_bf16_16816(ac[2 * np], a0, a1, a2, a3, b0, b1);
              mma_bf16_16816(ac[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
          }
        };
        {
          // two k-steps per iteration into independent accumulators (overlaps the MMA latency)
          float ac2[NT][4];
  #pragma unroll
          for (int n = 0; n < NT; ++n)
  #pragma unroll
            for (int e = 0; e < 4; ++e) ac2[n][e] = 0.f;
          int ks = warp;
          for (; ks + kCW < nk16; ks += 2 * kCW) {
            step(ks, acc);
            step(ks + kCW, ac2);
          }
          if (ks < nk16) step(ks, acc);
  #pragma unroll
          for (int n = 0; n < NT; ++n)
  #pragma unroll
            for (int e = 0; e < 4; ++e) acc[n][e] += ac2[n][e];
        }
        if ((len & 8) && warp == (nk16 % kCW)) {
          // tail of 8 rows (h_in is a multiple of 8): m16n8k8
          const int kb = nk16 * 16;
          const uint16_t* Xs = reinterpret_cast<const uint16_t*>(st_base + Cfg::kPartBytes);
          const uint32_t a0 = g < tlen ? ld_shared_u32(Xs + g * Cfg::XP + kb + 2 * tig) : 0u;
          const uint32_t a1 = g + 8 < tlen ? ld_shared_u32(Xs + (g + 8) * Cfg::XP + kb + 2 * tig) : 0u;
          if constexpr (NT == 1) {
            uint32_t b0, b1;  // b1 (lanes 8-15's rows) is not used
            ldsm_x2_trans(a_base + static_cast<uint32_t>(kb + lr) * (R * 2), b0, b1);
            mma_bf16_1688(acc[0], a0, a1, b0);
          } else {
  #pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              // matrices: (k 0-7, n 0-7), (k 0-7, n 8-15) of the pair
              const uint32_t addr = swz<Cfg::SWM>(a_base + static_cast<uint32_t>(kb + lr) * (R * 2) +
                                                  static_cast<uint32_t>(np * 16 + (lm & 1) * 8) * 2);
              uint32_t b0, b1;
              ldsm_x2_trans(addr, b0, b1);
              mma_bf16_1688(acc[2 * np], a0, a1, b0);
              mma_bf16_1688(acc[2 * np + 1], a0, a1, b1);
            }
          }
        }
        if (!(kind & kStLast)) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[slot]);  // header and data of this slot no longer read
        } else {
          // the slot is released before the exchange, so the producer keeps streaming
          int tokr[T];
  #pragma unroll
          for (int t = 0; t < T; ++t) tokr[t] = h.tok[t];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[slot]);
          // ---- this warp's partial v to shared memory, then the sum over warps
  #pragma unroll
          for (int n = 0; n < NT; ++n) {
            if (g < T) {
              red[warp][g][n * 8 + 2 * tig] = acc[n][0];
              red[warp][g][n * 8 + 2 * tig + 1] = acc[n][1];
            }
            if (g + 8 < T) {
              red[warp][g + 8][n * 8 + 2 * tig] = acc[n][2];
              red[warp][g + 8][n * 8 + 2 * tig + 1] = acc[n][3];
            }
          }
          if (!consumer_sync(&sm.abort)) {
            quit = true;
            return;
          }
          constexpr int kV4 = T * R / 4;  // float4 elements of one partial v
          auto red_sum = [&](int i) {
            float4 vp = make_float4(0.f, 0.f, 0.f, 0.f);
  #pragma unroll
            for (int w = 0; w < kCW; ++w) {
              const float4 u = reinterpret_cast<const float4*>(&red[w][0][0])[i];
              vp.x += u.x;
              vp.y += u.y;
              vp.z += u.z;
              vp.w += u.w;
            }
            return vp;
          };
          if (xchg) {
            if (!start_waited) {
              cluster_wait_acquire();  // every peer's mbarriers are initialised
              start_waited = true;
            }
            const uint32_t bar = smem_u32(&sm.xbar[b]);
            for (int i = ct; i < kV4; i += kCThreads) {
              const float4 vp = red_sum(i);
              reinterpret_cast<float4*>(&xbuf[b][rank][0][0])[i] = vp;
              const uint32_t src = smem_u32(&xbuf[b][rank][0][0]) + i * 16;
              for (int qq = 0; qq < C; ++qq)
                if (qq != rank && !(rank == 1 && withhold(2)))
                  st_async_v4(mapa_shared(src, qq), vp, mapa_shared(bar, qq));
            }
            bool got = true;
            if (lane == 0) got = mbar_wait(&sm.xbar[b], (nx >> 1) & 1, kWaitLimitNs);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
              give_up();
              return;
            }
            xarm = -1;
            // our own partial (plain stores) is visible to every consumer
            if (!consumer_sync(&sm.abort)) {
              quit = true;
              return;
            }
            for (int i = ct; i < kV4; i += kCThreads) {
              float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int qq = 0; qq < C; ++qq) {  // fixed order: identical v in every CTA
                const float4 u = reinterpret_cast<const float4*>(&xbuf[b][qq][0][0])[i];
                sum.x += u.x;
                sum.y += u.y;
                sum.z += u.z;
                sum.w += u.w;
              }
              reinterpret_cast<float4*>(&vfull[0][0])[i] = sum;
            }
          } else {
            for (int i = ct; i < kV4; i += kCThreads) reinterpret_cast<float4*>(&vfull[0][0])[i] = red_sum(i);
          }
          if (!consumer_sync(&sm.abort)) {
            quit = true;
            return;
          }
          ++nx;
          if (MODE == kModeShrink && rank == 0) {
            for (int idx = ct; idx < tlen * R; idx += kCThreads) {
              const int t = idx / R, k = idx % R;
              int tkv = -1;
  #pragma unroll
              for (int u = 0; u < T; ++u)
                if (u == t) tkv = tokr[u];
              if (tkv >= 0) q.v_out[static_cast<int64_t>(tkv) * R + k] = vfull[t][k];
            }
          }
        }
      } else {
        // ---- expand stage: y[tok, off .. off+len) += s * vfull[t] . B[:, off .. off+len)
        if (kind & kStFirst) {
          if (MODE == kModeExpand) {
            // every warp is done with the previous item's v
            if (!consumer_sync(&sm.abort)) {
              quit = true;
              return;
            }
            for (int idx = ct; idx < T * R; idx += kCThreads) {
              const int t = idx / R, k = idx % R;
              const int tk = t < tlen ? h.tok[t] : -1;
              vfull[t][k] = tk >= 0 ? q.v_in[static_cast<int64_t>(tk) * R + k] : 0.f;
            }
            if (!consumer_sync(&sm.abort)) {
              quit = true;
              return;
            }
          }
          // v as bf16 hi/lo MMA A fragments (rows >= tlen are zero)
          auto split = [&](int row, int col, uint32_t& hi, uint32_t& lo) {
            const bool ok = row < tlen;
            const float x0 = ok ? vfull[row][col] : 0.f, x1 = ok ? vfull[row][col + 1] : 0.f;
            hi = pack_bf16(x0, x1);
            const float2 hf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
            lo = pack_bf16(x0 - hf.x, x1 - hf.y);
          };
          if constexpr (Cfg::KS == 0) {
            split(g, 2 * tig, v8h[0], v8l[0]);
            split(g + 8, 2 * tig, v8h[1], v8l[1]);
          } else {
  #pragma unroll
            for (int ks = 0; ks < Cfg::KS; ++ks) {
              split(g, ks * 16 + 2 * tig, vah[ks][0], val[ks][0]);
              split(g + 8, ks * 16 + 2 * tig, vah[ks][1], val[ks][1]);
              split(g, ks * 16 + 8 + 2 * tig, vah[ks][2], val[ks][2]);
              split(g + 8, ks * 16 + 8 + 2 * tig, vah[ks][3], val[ks][3]);
            }
          }
        }
        const CCProj& pr = q.proj[pj];
        const float scale = pr.scale;
        uint16_t* const yg = pr.y;
        const int64_t ldy = pr.ldy;
        const int bw = h.pitch;  // box width (columns) of the B part; box = [R][bw]
        const uint32_t b_base = smem_u32(st_base);
        uint16_t* const Ys = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(st_base) + Cfg::kPartBytes);
        const int ntl = len >> 3;  // 8-column n-tiles in the stage
        const int tpb = bw >> 3;   // n-tiles per box (odd)
        const uint32_t mtpb = 65536u / static_cast<uint32_t>(tpb) + 1u;  // i / tpb == (i * mtpb) >> 16 here
        // element offset in the B part of column 0 of n-tile i (box-major layout [box][R][bw])
        auto tile_off = [&](int i) -> int {
          const int bx = static_cast<int>((static_cast<uint32_t>(i) * mtpb) >> 16);
          return bx * (R * bw) + (i - bx * tpb) * 8;
        };
        // y += s * products, in place in the stage's y rows (rows g, g+8 of a tile pair)
        auto upd = [&](int row, int col, float e0, float e1) {
          uint32_t* yp = reinterpret_cast<uint32_t*>(Ys + row * Cfg::XP + col);
          const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(yp));
          *yp = pack_bf16(yf.x + scale * e0, yf.y + scale * e1);
        };
        auto pair = [&](int j, float (&d0)[4], float (&d1)[4]) {
          // n-tiles j and j+1 (a missing second tile repeats the first)
          const int oa = tile_off(j), ob = j + 1 < ntl ? tile_off(j + 1) : oa;
  #pragma unroll
          for (int e = 0; e < 4; ++e) d0[e] = d1[e] = 0.f;
          if constexpr (Cfg::KS == 0) {
            // r = 8: matrices (k 0-7, tile a), (k 0-7, tile b); lanes 16+ repeat 0-15
            const int o = (lm & 1) ? ob : oa;
            uint32_t b0, b1;
            ldsm_x2_trans(b_base + static_cast<uint32_t>(o + lr * bw) * 2, b0, b1);
            mma_bf16_1688(d0, v8h[0], v8h[1], b0);
            mma_bf16_1688(d0, v8l[0], v8l[1], b0);
            mma_bf16_1688(d1, v8h[0], v8h[1], b1);
            mma_bf16_1688(d1, v8l[0], v8l[1], b1);
          } else {
            const int o = (lm >> 1) ? ob : oa;
  #pragma unroll
            for (int ks = 0; ks < Cfg::KS; ++ks) {
              // matrices: (k 0-7, a), (k 8-15, a), (k 0-7, b), (k 8-15, b)
              const int krow = ks * 16 + (lm & 1) * 8 + lr;
              uint32_t b0, b1, b2, b3;
              ldsm_x4_trans(b_base + static_cast<uint32_t>(o + krow * bw) * 2, b0, b1, b2, b3);
              mma_bf16_16816(d0, vah[ks][0], vah[ks][1], vah[ks][2], vah[ks][3], b0, b1);
              mma_bf16_16816(d0, val[ks][0], val[ks][1], val[ks][2], val[ks][3], b0, b1);
              mma_bf16_16816(d1, vah[ks][0], vah[ks][1], vah[ks][2], vah[ks][3], b2, b3);
              mma_bf16_16816(d1, val[ks][0], val[ks][1], val[ks][2], val[ks][3], b2, b3);
            }
          }
        };
        auto store = [&](int j, const float (&d0)[4], const float (&d1)[4]) {
          const bool has_b = j + 1 < ntl;
          const int col_a = 8 * j + 2 * tig, col_b = col_a + 8;
          if (g < tlen) {
            upd(g, col_a, d0[0], d0[1]);
            if (has_b) upd(g, col_b, d1[0], d1[1]);
          }
          if (g + 8 < tlen) {
            upd(g + 8, col_a, d0[2], d0[3]);
            if (has_b) upd(g + 8, col_b, d1[2], d1[3]);
          }
        };
        // this warp's tile pairs: j = 2*warp + 2*kCW*i, two pairs per iteration
        int j = 2 * warp;
        for (; j + 2 * kCW < ntl; j += 4 * kCW) {
          float d0[4], d1[4], d2[4], d3[4];
          pair(j, d0, d1);
          pair(j + 2 * kCW, d2, d3);
          store(j, d0, d1);
          store(j + 2 * kCW, d2, d3);
        }
        if (j < ntl) {
          float d0[4], d1[4];
          pair(j, d0, d1);
          store(j, d0, d1);
        }
        fence_proxy_async_smem();  // our y updates, visible to the bulk stores below
        if (!consumer_sync(&sm.abort)) {
          quit = true;
          return;
        }
        // ---- the tile's updated y rows back to global memory, one bulk copy per token
        if (ct < tlen) {
          const int tkv = h.tok[ct];
          if (tkv >= 0) {
            bulk_s2g(yg + static_cast<int64_t>(tkv) * ldy + off, Ys + ct * Cfg::XP, static_cast<uint32_t>(len) * 2u);
            bulk_commit();
            bulk_wait_read0();  // the slot may be refilled once the copy has read it
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }
    });
    if (quit) break;
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (xchg) {
    if (!start_waited) cluster_wait_acquire();
    // an exchange left before its peers' partials were in: their pushes may
    // still arrive, and must land before this CTA may leave (bounded)
    if (xarm >= 0 && lane == 0) (void)mbar_wait(&sm.xbar[xarm], (nx >> 1) & 1, kWaitLimitNs);
    // no CTA leaves while a peer may still push into its shared memory
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
}

// ------------------------------------------------------------------ host side

namespace {

struct KernelInfo {
  int max_groups = 0;  // co-resident clusters (or CTA groups) on the device
};

// One-launch step limits (build-time knobs, set by measurement): the sort's
// temporaries (n + P + 1 ints) fit ring stage 0, and its result (permutation,
// offsets, adapters, count) adds at most kSegExtraMaxBytes of shared memory
// per CTA, small enough to keep the CTAs per SM of the decode shapes.
#ifndef LSG_SEG_IN_KERNEL_MAX_TOKENS
#define LSG_SEG_IN_KERNEL_MAX_TOKENS 128
#endif
#ifndef LSG_SEG_IN_KERNEL_MAX_ADAPTERS
#define LSG_SEG_IN_KERNEL_MAX_ADAPTERS 1024
#endif
constexpr int kSegInKernelMaxTokens = LSG_SEG_IN_KERNEL_MAX_TOKENS;
constexpr int kSegInKernelMaxAdapters = LSG_SEG_IN_KERNEL_MAX_ADAPTERS;
constexpr size_t kSegExtraMaxBytes = 2 * 1024;
size_t seg_extra_bytes(int n, int P) {
  const int ms = std::min(n, P);
  return static_cast<size_t>(n + (ms + 1) + std::max(ms, 1) + 1) * sizeof(int32_t);
}
static_assert((LSG_SEG_IN_KERNEL_MAX_TOKENS * 3 + 3) * 4 <= kSegExtraMaxBytes, "segmentation result size");
static_assert((LSG_SEG_IN_KERNEL_MAX_TOKENS + LSG_SEG_IN_KERNEL_MAX_ADAPTERS + 1) * 4 <= LSG_CC_KB_R8 * 1024,
              "sort temporaries in ring stage 0 (rank 8)");
static_assert((LSG_SEG_IN_KERNEL_MAX_TOKENS + LSG_SEG_IN_KERNEL_MAX_ADAPTERS + 1) * 4 <= LSG_CC_KB_SMALL * 1024,
              "sort temporaries in ring stage 0");

// Stage shape of rank r in the ring of a kernel whose largest rank is RM.
struct RankShape {
  int BA, WS, SWA;
};
template <int T, int RM>
RankShape rank_shape(int r) {
  switch (r) {
    case 8: return {CCCfg<8, T, RM>::BA, CCCfg<8, T, RM>::WS, CCCfg<8, T, RM>::SWA};
    case 16: return {CCCfg<16, T, RM>::BA, CCCfg<16, T, RM>::WS, CCCfg<16, T, RM>::SWA};
    case 32: return {CCCfg<32, T, RM>::BA, CCCfg<32, T, RM>::WS, CCCfg<32, T, RM>::SWA};
    default: return {CCCfg<64, T, RM>::BA, CCCfg<64, T, RM>::WS, CCCfg<64, T, RM>::SWA};
  }
}

// Encodes the tensor-map pairs of every (projection, rank of `ranks`) and
// launches.  prm.t holds the projections, the tables and rmax / n_slots.
template <int RSET, int T, int MODE>
lora_status launch_rtm(CCParams& prm, const int* ranks, int n_ranks, int items_bound, size_t extra_smem,
                       cudaStream_t stream) {
  constexpr int RM = set_max_rank(RSET);
  auto kern = sgmv_cc_kernel<RSET, T, MODE>;
  const size_t smem = sizeof(CCSmem<RM, T>) + extra_smem;
  // occupancy with the segmentation result rounded up to 256 bytes (cached per size class)
  const int var = static_cast<int>((extra_smem + 255) / 256);
  const size_t smem_occ = sizeof(CCSmem<RM, T>) + static_cast<size_t>(var) * 256;
  if (extra_smem > kSegExtraMaxBytes) return LORA_ERR_UNSUPPORTED;
  const int C = prm.t.csplit;
  const bool cluster = (MODE & kModeShrink) && C > 1;
  if (prm.t.n_proj * n_ranks > kMaxProj) return LORA_ERR_UNSUPPORTED;

  prm.t.rank_mask = 0;
  for (int j = 0; j < n_ranks; ++j) {
    if ((rank_bit(ranks[j]) & RSET) == 0) return LORA_ERR_UNSUPPORTED;
    prm.t.rank_mask |= rank_bit(ranks[j]);
  }
  int m = 0;
  for (int i = 0; i < prm.t.n_proj; ++i) {
    CCProj& q = prm.t.proj[i];
    for (int c = 0; c < 4; ++c) prm.t.map_of[i][c] = -1;
    for (int j = 0; j < n_ranks; ++j, ++m) {
      const int r = ranks[j];
      const RankShape sh = rank_shape<T, RM>(r);
      prm.t.map_of[i][rank_class(r)] = m;
      prm.t.map_bw[m] = 8;
      prm.t.map_nb[m] = 1;
      if (MODE & kModeShrink) {
        const uint64_t rows = static_cast<uint64_t>(prm.t.n_slots) * q.h_in * (prm.t.rmax / r);
        const uint64_t dims[2] = {static_cast<uint64_t>(r), rows};
        const uint64_t strides[1] = {static_cast<uint64_t>(r) * 2};
        const uint32_t box[2] = {static_cast<uint32_t>(r), static_cast<uint32_t>(sh.BA)};
        const lora_status s = encode_tmap_bf16(&prm.tmA[m], q.A, 2, dims, strides, box, sh.SWA);
        if (s != LORA_OK) return s;
      }
      if (MODE & kModeExpand) {
        // stage = nb boxes of bw columns, nb*bw <= WS; bw <= 256 (the TMA box
        // limit) and an odd multiple of 8 (16-byte chunks), which puts the 8 rows
        // an ldmatrix reads into different banks.  Fewest boxes that cover a
        // stage's share of the chunk.
        const int nst = std::max(1, ceil_div(q.n_chunk, sh.WS));
        const int pe = round_up(ceil_div(q.n_chunk, nst), 8);
        int bw = 8, nb = 0;
        for (int k = 1; k <= 16 && nb == 0; ++k) {
          int w = round_up(ceil_div(pe, k), 8);
          if ((w / 8) % 2 == 0) w += 8;
          if (w <= 256 && k * w <= sh.WS) {
            nb = k;
            bw = w;
          }
        }
        if (nb == 0) {  // covering is impossible within WS: largest odd box that fits
          nb = 1;
          bw = std::min(256, sh.WS) / 8 * 8;
          if ((bw / 8) % 2 == 0) bw -= 8;
        }
        prm.t.map_bw[m] = bw;
        prm.t.map_nb[m] = nb;
        const uint64_t dims[2] = {static_cast<uint64_t>(q.h_out), static_cast<uint64_t>(prm.t.n_slots) * prm.t.rmax};
        const uint64_t strides[1] = {static_cast<uint64_t>(q.h_out) * 2};
        const uint32_t box[2] = {static_cast<uint32_t>(bw), static_cast<uint32_t>(r)};
        const lora_status s = encode_tmap_bf16(&prm.tmB[m], q.B, 2, dims, strides, box, 0);
        if (s != LORA_OK) return s;
      }
    }
  }

  static std::mutex mu;
  static KernelInfo info[64][kMaxC + 1][kSegExtraMaxBytes / 256 + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  KernelInfo ki;
  {
    std::lock_guard<std::mutex> lk(mu);
    ki = info[dev & 63][C][var];
  }
  if (ki.max_groups == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(CCSmem<RM, T>) + kSegExtraMaxBytes)) != cudaSuccess)
      return LORA_ERR_CUDA;
    if (cluster) {
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute at[1];
      cfg.gridDim = dim3(C * 1024);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem_occ;
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = C;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) return LORA_ERR_CUDA;
      ki.max_groups = std::max(1, nclusters);
    } else {
      int per_sm = 0, nsm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_occ) != cudaSuccess)
        return LORA_ERR_CUDA;
      if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LORA_ERR_CUDA;
      ki.max_groups = std::max(1, per_sm * nsm / C);
    }
    std::lock_guard<std::mutex> lk(mu);
    info[dev & 63][C][var] = ki;
  }
  const int groups = std::max(1, std::min(items_bound, ki.max_groups));

  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[2];
  int na = 0;
  cfg.gridDim = dim3(groups * C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  if (cluster) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = C;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, prm));
}

template <int R, int T>
lora_status dispatch_mode(Mode m, CCParams& prm, int items_bound, size_t extra, cudaStream_t st) {
  const int ranks[1] = {R};
  switch (m) {
    case kModeShrink: return launch_rtm<rank_bit(R), T, kModeShrink>(prm, ranks, 1, items_bound, 0, st);
    case kModeExpand: return launch_rtm<rank_bit(R), T, kModeExpand>(prm, ranks, 1, items_bound, 0, st);
    default: return launch_rtm<rank_bit(R), T, kModeFused>(prm, ranks, 1, items_bound, extra, st);
  }
}

template <int T>
lora_status dispatch_r(int r, Mode m, CCParams& prm, int items_bound, size_t extra, cudaStream_t st) {
  switch (r) {
    case 8: return dispatch_mode<8, T>(m, prm, items_bound, extra, st);
    case 16: return dispatch_mode<16, T>(m, prm, items_bound, extra, st);
    case 32: return dispatch_mode<32, T>(m, prm, items_bound, extra, st);
    case 64: return dispatch_mode<64, T>(m, prm, items_bound, extra, st);
    default: return LORA_ERR_UNSUPPORTED;
  }
}

// Mixed ranks (fused only): one launch per group of projections whose
// (projection, rank) map pairs fit the parameter block.
template <int T>
lora_status dispatch_mixed(CCParams& base, const int* ranks, int n_ranks, int items_per_proj, cudaStream_t st) {
  const int per = std::max(1, kMaxProj / n_ranks);
  const int n_proj = base.t.n_proj;
  for (int p0 = 0; p0 < n_proj; p0 += per) {
    CCParams prm = base;
    const int np = std::min(per, n_proj - p0);
    for (int i = 0; i < np; ++i) prm.t.proj[i] = base.t.proj[p0 + i];
    prm.t.n_proj = np;
    const int items = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(items_per_proj) * np, 1 << 30));
    const lora_status s = launch_rtm<kAllRanks, T, kModeFused>(prm, ranks, n_ranks, items, 0, st);
    if (s != LORA_OK) return s;
  }
  return LORA_OK;
}

}  // namespace

lora_status launch_sgmv_cc(const SgmvCall& call, cudaStream_t stream) {
  const int n = call.seg.n_tokens;
  const int S_max = call.seg.max_segments;
  int hmax = 0;
  for (int i = 0; i < call.n_proj; ++i) {
    if (call.mode & kModeShrink) hmax = std::max(hmax, call.proj[i].h_in);
    if (call.mode & kModeExpand) hmax = std::max(hmax, call.proj[i].h_out);
  }
  // ranks per item: about LSG_CC_ROWS_PER_CTA rows/columns per CTA, at most 8 (portable cluster)
  const int C = std::clamp(ceil_div(hmax, LSG_CC_ROWS_PER_CTA), 1, kMaxC);
  // tokens per tile (MMA rows): small tiles when segments are short on average
  const double avg = static_cast<double>(n) / std::max(1, std::min(n, call.n_adapters));
  const int T = avg <= LSG_CC_T4_MAX_AVG ? 4 : 16;

  CCParams prm{};
  for (int i = 0; i < call.n_proj; ++i) {
    const ProjArgs& a = call.proj[i];
    CCProj& q = prm.t.proj[i];
    q.x = a.x;
    q.A = a.A;
    q.B = a.B;
    q.y = a.y;
    q.ldx = a.ldx;
    q.ldy = a.ldy;
    q.h_in = a.h_in;
    q.h_out = a.h_out;
    q.k_chunk = round_up(ceil_div(a.h_in, C), 16);
    q.n_chunk = round_up(ceil_div(a.h_out, C), 8);
    q.scale = a.scale;
  }
  prm.t.perm = call.seg.perm;
  prm.t.seg_offsets = call.seg.seg_offsets;
  prm.t.seg_adapter = call.seg.seg_adapter;
  prm.t.num_segments = call.seg.num_segments;
  prm.t.v_out = call.v_out;
  prm.t.v_in = call.v_in;
  prm.t.err_flag = call.err_flag;
  prm.t.n_proj = call.n_proj;
  prm.t.n_tokens = n;
  prm.t.max_segments = S_max;
  prm.t.n_adapters = call.n_adapters;
  prm.t.csplit = C;
  prm.t.skip_long = 0;
  const bool slots = call.slot_of != nullptr;
  prm.t.slot_of = call.slot_of;
  prm.t.rank_of = call.rank_of;
  prm.t.n_slots = slots ? call.n_slots : call.n_adapters;
  prm.t.rmax = slots ? call.r_max : call.r;
  const bool tc = !call.long_done && sgmv_tc_applicable(call);
  size_t extra = 0;
  if (call.ids != nullptr) {
    // segmentation first: inside this launch when it fits, else its own kernel
    if (!slots && !tc && call.mode == kModeFused && n <= kSegInKernelMaxTokens &&
        call.n_adapters <= kSegInKernelMaxAdapters) {
      prm.t.ids = call.ids;
      extra = seg_extra_bytes(n, call.n_adapters);
      if (call.ids_host != nullptr) {
        static_assert(kIdsInParamsMax >= LSG_SEG_IN_KERNEL_MAX_TOKENS, "ids in the parameters");
        std::memcpy(prm.ids_in_params, call.ids_host, static_cast<size_t>(n) * sizeof(int32_t));
        prm.n_ids_in_params = n;
      }
    } else {
      if (call.ids_host != nullptr &&
          cudaMemcpyAsync(const_cast<int32_t*>(call.ids), call.ids_host, static_cast<size_t>(n) * sizeof(int32_t),
                          cudaMemcpyDefault, stream) != cudaSuccess)
        return LORA_ERR_CUDA;
      const lora_status s = launch_segment(call.ids, n, call.n_adapters, const_cast<int32_t*>(call.seg.perm),
                                           const_cast<int32_t*>(call.seg.seg_offsets),
                                           const_cast<int32_t*>(call.seg.seg_adapter),
                                           const_cast<int32_t*>(call.seg.num_segments), call.seg_hist,
                                           call.err_flag, stream);
      if (s != LORA_OK) return s;
    }
  }
  if (call.long_done) {
    prm.t.skip_long = 1;  // another launch took the long segments
  } else if (tc && !slots) {
    // long segments on tcgen05 tiles, the rest of the batch here
    const lora_status s = launch_sgmv_tc(call, stream);
    if (s != LORA_OK) return s;
    prm.t.skip_long = 1;
  } else if (tc && slots) {
    // one tensor-tile launch per rank of the mask
    for (int r = 8; r <= 64; r *= 2) {
      if (!(call.rank_mask & static_cast<unsigned>(rank_bit(r)) ) || r > call.r_max) continue;
      SgmvCall cr = call;
      cr.r = r;
      const lora_status s = launch_sgmv_tc(cr, stream);
      if (s != LORA_OK) return s;
      prm.t.tc_ranks |= rank_bit(r);
    }
    prm.t.skip_long = prm.t.tc_ranks != 0;
  }

  // upper bound of the number of tiles: sum over segments of ceil(len/T)
  const int64_t tiles = std::min<int64_t>(n, (static_cast<int64_t>(n) + static_cast<int64_t>(S_max) * (T - 1)) / T);
  int ranks[4], n_ranks = 0;
  if (slots) {
    for (int c = 0; c < 4; ++c)
      if (call.rank_mask & (1u << c)) ranks[n_ranks++] = 8 << c;
  }
  if (slots && n_ranks > 1) {
    if (call.mode != kModeFused) return LORA_ERR_UNSUPPORTED;
    const int items_per_proj = static_cast<int>(std::min<int64_t>(tiles, 1 << 30));
    if (T == 4) return dispatch_mixed<4>(prm, ranks, n_ranks, items_per_proj, stream);
    return dispatch_mixed<16>(prm, ranks, n_ranks, items_per_proj, stream);
  }
  const int r = slots ? ranks[0] : call.r;
  const int items_bound = static_cast<int>(std::min<int64_t>(tiles * call.n_proj, 1 << 30));
  if (T == 4) return dispatch_r<4>(r, call.mode, prm, items_bound, extra, stream);
  return dispatch_r<16>(r, call.mode, prm, items_bound, extra, stream);
}

}  // namespace lsg
