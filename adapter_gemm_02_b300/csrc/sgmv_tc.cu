// SGMV for long segments (prefill) on the 5th-generation tensor cores.
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Key
// points": the SGMV kernel batches the LoRA add-on computation across
// adapters and uses the GPU's tensor cores; "Interesting ideas" I2: sorting
// the batch by adapter turns scattered small products into dense segments.
// For a prefill segment (hundreds of tokens of one adapter) both products
// are real matrix products, tiled here as M = 128 tokens:
//
//   shrink  v[128][r]   = x[128][h_in] . A[h_in][r]            (K = h_in)
//   expand  y[128][c]  += s * v[128][r] . B[r][c], c in chunk  (K = r)
//
// One CTA per SM, persistent, twelve warps with fixed roles:
//   warps 0-3, 8-11  epilogue, two groups of four (warp w: TMEM lane quarter
//              w % 4).  Group 0 turns v (fp32, TMEM) into the expand's bf16
//              operand pair v = hi + lo, written back into TMEM (in shared
//              memory for the cluster variant, whose peers write it there);
//              both groups then add s * acc to their 32 columns of each
//              64-column y block in shared memory, and group 0 stores the
//              block (one TMA box per quarter)
//   warp 4     shrink producer: TMA x tiles [128][64] (K-major, 128 B swizzle)
//              and A tiles [64][r] (MN-major, 2r-byte swizzle), 6 stages
//   warp 5     expand producer: TMA B tiles [r][64] (MN-major) and y tiles
//              [128][64] (128 B swizzle) on separate barriers, in the stages
//              the rest of shared memory holds (3 at r = 64)
//   warp 6     TMEM allocation; one thread issues the shrink MMAs
//   warp 7     one thread issues the expand MMAs
//              (tcgen05.mma kind::f16, fp32 accumulators in TMEM: v in columns
//              0..r-1, two 64-column expand buffers, so the epilogue of one
//              block overlaps the MMAs of the next).  With one issuer per
//              stream the shrink of item i+1 streams x and A while item i is
//              expanded; the epilogue orders the two: it reads v(i) out of
//              TMEM before the shrink of item i+1 may overwrite it (v_read),
//              and it rewrites the v operand only after the last expand MMAs
//              of item i completed.
//
// Work item = (128-token tile of a segment, projection, column chunk of
// h_out), dealt to the CTAs (or to clusters of C CTAs that share an item:
// split-K shrink, split-N expand, partial v summed through distributed
// shared memory) in a weighted round robin (TcSched).  Each item recomputes its tile's shrink (x is re-read from
// L2 by the items of the same tile), which keeps items of similar size for
// load balance.  Every segment of at least kLongSeg tokens is taken here (the
// decode kernel skips exactly these).  A tile whose rows are contiguous in
// x / y (a prefill request, or a run of one inside a segment of several
// requests) moves with 2-D tensor copies; any other tile (tokens of one
// adapter spread over the batch) gathers its rows through the permutation:
// the producer lanes copy x rows with 16-byte cp.async copies and load y rows
// four at a time by tile::gather4 tensor copies into the swizzled tile, and
// the updated y rows go back by tile::scatter4 tensor stores (rows of an
// incomplete group of four by 16-byte stores).
// Gathered tiles run at about half the rate of contiguous ones: every 128-byte
// row piece is its own request, against one 16 KB box.
//
// Rank 8 runs at an MMA width of 16: the shrink's N = 16 columns read the A
// tile's 8 columns plus 8 columns of other shared memory, whose results are
// never used; the expand's K = 16 takes v with columns 8..15 zero and a B
// tile whose rows 8..15 are a zero block that no copy writes.
//
// Modes: fused (v stays on chip), shrink (v written to device memory in fp32,
// token order), expand (v read from device memory).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace lsg {

constexpr int kTcThreads = 384;
constexpr int kTcEpiThreads = 128;  // one epilogue group: 4 warps, one per TMEM lane quarter
// Shrink ring depth: the shrink streams from L2 (and DRAM) with a latency of
// microseconds, so its ring sets its rate.  Rank 64, 13B layer: 4 / 5 / 6 / 7
// shrink stages (the expand ring takes the rest: 5 / 4 / 3 / 2) 415 / 393 /
// 391 / 508 us.
#ifndef LSG_TC_SH_STAGES
#define LSG_TC_SH_STAGES 6
#endif
#ifndef LSG_TC_CHUNK
#define LSG_TC_CHUNK 5120
#endif
#ifndef LSG_TC_BN
#define LSG_TC_BN 64
#endif
constexpr int kShStages = LSG_TC_SH_STAGES;
constexpr int kBN = LSG_TC_BN;       // expand block columns (MMA N): 64 (128 leaves the cluster ring one stage: rejected below)
constexpr int kBH = kBN / 64;        // 64-column halves per block
static_assert(kBN == 64, "expand block: two epilogue groups of 32 columns");
#ifndef LSG_TC_EX_STAGES
#define LSG_TC_EX_STAGES 4
#endif
constexpr int kExStages = LSG_TC_EX_STAGES;
// the cluster variant's rings (its partial-v receive buffer takes their room)
#ifndef LSG_TC_SH_STAGES_CL
#define LSG_TC_SH_STAGES_CL 3
#endif
#ifndef LSG_TC_EX_STAGES_CL
#define LSG_TC_EX_STAGES_CL 3
#endif
// Gathered tiles' rows, for the shrink's x and the expand's y apart: 1 =
// four-row tensor gathers (one per lane and stage), 0 = 16-byte cp.async
// copies by the producer's lanes.  The full 13B prefill layer with
// interleaved requests: x by cp.async and y by gathers 755 us, both by
// gathers 805 us, x by gathers and y by cp.async 800 us, both by cp.async
// 849 us (the tensor-copy unit issues every 128-byte row piece of a gather
// as its own request; the copies split the pieces between it and the
// load/store units).
#ifndef LSG_TC_GATHER4_X
#define LSG_TC_GATHER4_X 0
#endif
#ifndef LSG_TC_GATHER4_Y
#define LSG_TC_GATHER4_Y 1
#endif
// Gathered tiles' updated y rows: 1 = four-row tensor scatters, 0 = 16-byte
// stores by the epilogue threads.
#ifndef LSG_TC_SCATTER4
#define LSG_TC_SCATTER4 1
#endif
// 1: the expand's A operand (v as a bf16 hi / lo pair) lives in TMEM, which
// frees its shared memory for expand ring stages; 0: in shared memory.  The
// cluster variant keeps it in shared memory (peers write it there).
#ifndef LSG_TC_VOP_TMEM
#define LSG_TC_VOP_TMEM 1
#endif
// most expand ring stages (the ring takes what shared memory is left, up to this)
#ifndef LSG_TC_EX_STAGES_MAX
#define LSG_TC_EX_STAGES_MAX 8
#endif
// 1: heavy item slots (see TcSched) go to the groups with one item fewer.
#ifndef LSG_TC_HEAVY_FIRST
#define LSG_TC_HEAVY_FIRST 1
#endif
// Item cost model: us per shrink k-block and per expand block.  Fitted to
// the 4-stage shrink ring (50-57 us of shrink over 80 k-blocks, 137-141 us
// over 216, 67-78 us of expand over 72-80 blocks) and kept, by measurement:
// with the 6-stage ring the items measure 38-40 / 103 / 77-98 us, but a fit
// to those (0.48, 1.05) no longer marks the 13B down projection heavy and the
// layer takes 415 instead of 390 us (the 2-request batch 244 instead of 216).
#ifndef LSG_TC_COST_KB
#define LSG_TC_COST_KB 0.7
#endif
#ifndef LSG_TC_COST_BLK
#define LSG_TC_COST_BLK 0.95
#endif
// 1: heavy items start at pass 1 of the round robin (after each group's
// first light item).
#ifndef LSG_TC_HEAVY_LATE
#define LSG_TC_HEAVY_LATE 1
#endif
// 1: an expand slot goes back as soon as this block's y stores have read it;
// 0: one block later (after the next block's stores are issued).
#ifndef LSG_TC_RELEASE_EARLY
#define LSG_TC_RELEASE_EARLY 1
#endif

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemV = 0;      // v accumulator: columns [0, r)
constexpr uint32_t kTmemAcc = 128;  // expand accumulators: [128, 256), [256, 384)
constexpr uint32_t kTmemVop = 384;  // (operand in TMEM) v as bf16 hi [384, 384 + r/2), lo [.., 384 + r)
constexpr int kChunkCols = LSG_TC_CHUNK;  // expand columns per item, about
constexpr int kMaxItemsPerTile = 64;
constexpr int kMaxC = 8;  // CTAs per cluster (portable limit)
constexpr uint64_t kTcWaitNs = LSG_WAIT_LIMIT_NS;

#ifdef LSG_TEST_HOOKS
__device__ int g_test_withhold;
__device__ __forceinline__ bool withhold(int what) { return *(volatile int*)&g_test_withhold == what; }
lora_status test_withhold_tc(int what) { return cuda_status(cudaMemcpyToSymbol(g_test_withhold, &what, sizeof(int))); }
#else
__device__ __forceinline__ bool withhold(int) { return false; }
#endif

struct TcProj {
  const uint16_t* x;  // gathered tiles' x rows (copied by the producer)
  int64_t ldx;
  uint16_t* y;  // gathered tiles' y rows, and the direct stores of a tile's last rows
  int64_t ldy;
  int32_t h_in, h_out;
  int32_t chunk;  // columns per chunk (multiple of 128)
  float scale;
};

struct TcTail {
  TcProj proj[kMaxProj];
  int8_t item_proj[kMaxItemsPerTile];
  int8_t item_chunk[kMaxItemsPerTile];
  int8_t slot_order[kMaxItemsPerTile];  // a tile's item slots, the n_heavy heavy ones first
  int32_t n_heavy;                      // heavy item slots per tile (0: plain round robin)
  const int32_t* perm;
  const int32_t* seg_offsets;
  const int32_t* seg_adapter;
  const int32_t* num_segments;
  int32_t* err_flag;
  float* v_out;       // shrink mode: v [n][r] fp32, token order
  const float* v_in;  // expand mode
  int32_t n_proj;
  int32_t ipt;  // items per tile
  int32_t n_tokens;
  int32_t max_segments;
  int32_t n_adapters;
  int32_t csplit;  // CTAs per item (cluster size C): split-K shrink, split-N expand
  int32_t kparts;  // shrink mode: items per (tile, projection), each a part of the k-blocks;
                   // part p writes its partial v to v_out + p * n * r
  // Slot arenas (null slot_of: contiguous pool, slab = adapter id): a long
  // segment is taken when its adapter's slot is valid and its rank is this
  // kernel's rank; the slab index is then the slot.
  const int32_t* slot_of;
  const int32_t* rank_of;
  int32_t n_slabs;  // slabs in the pool / slots in the arenas
  int32_t rmax;     // B rows per slab (the contiguous pool: r)
  int32_t rank;     // this kernel's rank
};

struct TcParams {
  CUtensorMap tmX[kMaxProj];   // x [n][h_in], box {64, 128}, 128 B swizzle
  CUtensorMap tmXg[kMaxProj];  // x, box {64, 1} (four-row gathers), 128 B swizzle
  CUtensorMap tmA[kMaxProj];   // A slabs [n_slabs][h_in][r] (slab stride h_in*rmax), box {r, 64, 1}, 2r B swizzle
  CUtensorMap tmB[kMaxProj];   // B rows [n_slabs*rmax][h_out], box {64, r}, 128 B swizzle
  CUtensorMap tmYl[kMaxProj];  // y [n][h_out], box {64, 128}, 128 B swizzle (load)
  CUtensorMap tmYg[kMaxProj];  // y, box {64, 1} (four-row scatters), 128 B swizzle
  CUtensorMap tmYs[kMaxProj];  // y, box {64, 32}, 128 B swizzle (store)
  TcTail t;
};

template <int R>
struct TcCfg {
  static constexpr int RP = R < 16 ? 16 : R;                       // MMA width of the rank
  static constexpr int kShA = 64 * R * 2;                          // A tile bytes the copy writes
  static constexpr int kShARoom = 64 * RP * 2;                     // A tile bytes the shrink MMAs read
  static constexpr int kShBytes = ((16384 + kShARoom + 1023) / 1024) * 1024;
  static constexpr int kExY = 16384 * kBH;                         // y tile bytes [128][kBN]
  static constexpr int kExBCopy = R * 128 * kBH;                   // B tile bytes the copy writes
  static constexpr int kExB = RP * 128 * kBH;                      // B tile bytes the expand MMAs read
  static constexpr int kExBytes = ((kExY + kExB + 1023) / 1024) * 1024;
  static constexpr int kVop = 128 * RP * 2;                        // one bf16 operand [128][RP]
  static constexpr uint32_t kSwR = RP * 2;                         // swizzle span of RP-wide rows
  static constexpr uint32_t kSwM = kSwR / 16 - 1;
};

// Shared memory.  CL: the cluster variant, which adds the partial-v receive
// buffer and takes one stage from each ring to make room for it.
template <int R, bool CL>
struct TcSmem {
  static constexpr bool kVopT = LSG_TC_VOP_TMEM && !CL;  // operand pair in TMEM
  static constexpr int kVopBytes = kVopT ? 1024 : 2 * TcCfg<R>::kVop;
  static constexpr int kSh = CL ? LSG_TC_SH_STAGES_CL : kShStages;
  // non-cluster: as many expand stages as the rest of 227 KB holds (8 KB for
  // the tail and barriers), at least LSG_TC_EX_STAGES
  static constexpr int kExFit =
      (227 * 1024 - kSh * TcCfg<R>::kShBytes - kVopBytes - 8192) / TcCfg<R>::kExBytes;
  static constexpr int kEx = CL ? LSG_TC_EX_STAGES_CL
                                : (LSG_TC_VOP_TMEM ? (kExFit < LSG_TC_EX_STAGES_MAX ? kExFit : LSG_TC_EX_STAGES_MAX)
                                                   : kExStages);
  // the epilogue hands a slot back one block late, so each ring needs two
  // stages (an expand block of 128 columns leaves the cluster variant one)
  static_assert(kSh >= 2 && kEx >= 2, "ring depth");
  alignas(1024) uint8_t sh[kSh][TcCfg<R>::kShBytes];
  alignas(1024) uint8_t ex[kEx][TcCfg<R>::kExBytes];
  alignas(1024) uint8_t vop[kVopT ? 1 : 2][kVopT ? 1024 : TcCfg<R>::kVop];  // hi, lo (in shared memory)
  alignas(16) float rbuf[CL ? 128 * R : 4];      // partial v rows this CTA owns: [source rank][row][r]
  alignas(16) TcTail t;
  alignas(8) uint64_t sh_full[kSh];
  uint64_t sh_empty[kSh];
  uint64_t ex_full[kEx];  // B tile landed (the expand MMAs wait for it)
  uint64_t ey_full[kEx];  // y tile landed (the epilogue waits for it)
  uint64_t ex_empty[kEx];
  uint64_t v_full;     // shrink MMAs of the item done (v in TMEM)
  uint64_t v_read;     // the epilogue has read v out of TMEM
  uint64_t vop_ready;  // the v operand pair is complete in shared memory
  uint64_t rs_full;    // (cluster) every rank's partial of the rows this CTA owns has arrived
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain[2];  // each MMA issuer, at exit: its MMAs have completed
  uint32_t tmem_base;
  int32_t abort;
};

// One 128-token tile of a segment taken by this kernel.
struct TcTile {
  int t0;    // position of its first token in the permutation
  int tlen;  // tokens (<= 128)
  int a;     // slab (adapter id, or slot with slot arenas)
  int row;   // first x / y row when the tile's rows are contiguous, else -1 (rows through perm)
};

// Cursor over the segments taken by this kernel (at least kLongSeg tokens),
// 32 at a time, locating 128-token tiles.  Executed by a full warp; tile
// indices asked for only grow.
struct TcCursor {
  int base = 0, tiles_before = 0, S = 0;
  int off = 0, len = 0, ad = -1, row0 = -1;  // segment base + lane

  __device__ void load(const TcTail& q, int lane) {
    const int s = base + lane;
    off = 0;
    len = 0;
    ad = -1;
    row0 = -1;
    if (s < S) {
      const int o = q.seg_offsets[s];
      const int e = q.seg_offsets[s + 1];
      ad = q.seg_adapter[s];
      const int l = (o >= 0 && e <= q.n_tokens && e >= o) ? e - o : 0;
      if (l >= kLongSeg) {
        bool take = true;
        if (q.slot_of != nullptr) {
          // slot arenas: the slab is the slot; other ranks and invalid entries
          // stay with the split-K kernel
          int slab = -1;
          if (ad >= 0 && ad < q.n_adapters) {
            const int sl = q.slot_of[ad], rk = q.rank_of[ad];
            if (sl >= 0 && sl < q.n_slabs && rk == q.rank) slab = sl;
          }
          take = slab >= 0;
          ad = slab;
        }
        if (take) {
          off = o;
          len = l;
          // perm is ascending within a segment, so first and last rows l - 1
          // apart mean the rows are contiguous
          const int f = q.perm[o], b = q.perm[e - 1];
          if (f >= 0 && b < q.n_tokens && b - f == l - 1) row0 = f;
        }
      }
    }
  }

  __device__ void init(const TcTail& q, int lane) {
    S = min(max(*q.num_segments, 0), q.max_segments);
    load(q, lane);
  }

  __device__ bool find(const TcTail& q, int lane, int tile, TcTile& out) {
    if (tile < tiles_before) {  // an earlier tile: walk again from the first segment
      base = 0;
      tiles_before = 0;
      load(q, lane);
    }
    while (base < S) {
      const int tl = (len + 127) >> 7;
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
        const int l = __shfl_sync(0xffffffffu, len, ls);
        const int o = __shfl_sync(0xffffffffu, off, ls);
        const int r0 = __shfl_sync(0xffffffffu, row0, ls);
        out.a = __shfl_sync(0xffffffffu, ad, ls);
        const int k = (tile - tiles_before - excl) * 128;
        out.tlen = min(128, l - k);
        out.t0 = o + k;
        out.row = r0 >= 0 ? r0 + k : -1;
        if (r0 < 0) {
          // a segment of several runs of rows (requests of one adapter apart
          // in the batch): a tile inside one run still moves by 2-D tiles
          int f = -1, b = -1;
          if (lane == 0) {
            f = q.perm[out.t0];
            b = q.perm[out.t0 + out.tlen - 1];
          }
          f = __shfl_sync(0xffffffffu, f, 0);
          b = __shfl_sync(0xffffffffu, b, 0);
          if (f >= 0 && b < q.n_tokens && b - f == out.tlen - 1) out.row = f;
        }
        return true;
      }
      tiles_before += total;
      base += 32;
      load(q, lane);
    }
    return false;
  }
};

// The order of the launch's items.  Items are (tile, slot) pairs; group g
// takes the positions g, g + G, g + 2G, ... of a sequence.  Without heavy
// slots the sequence is the items in tile-major order (plain round robin).
// A tile's heavy slots (about twice the median item: a projection with a long
// shrink, such as the MLP down projection) weigh two positions: heavy item j
// takes position (h0 + 2 (j / G)) G + j mod G and the one a pass later in
// the same group, so a group with a heavy item takes one light item fewer.
// The light items fill the remaining positions in tile order.  The heavy
// passes start at pass h0 = 1 when every group has a light item for pass 0:
// a heavy item's long shrink then overlaps the expand of the group's first
// item instead of delaying the group's first expand.
struct TcSched {
  int L = 0x7fffffff, H = 0, G = 1, hr = 0, hrem = 0, h0 = 0, nh = 0, nl = 0;
  __device__ TcSched(const TcTail& q, TcCursor& cur, int lane, int groups) {
    G = groups;
    nh = q.n_heavy;
    if (nh == 0) return;
    TcTile t;
    (void)cur.find(q, lane, 0x7fffffff, t);  // walks every segment: the tile count
    const int nt = cur.tiles_before;
    nl = q.ipt - nh;
    H = nt * nh;
    L = nt * nl;
    hr = H / G;
    hrem = H - hr * G;
    h0 = LSG_TC_HEAVY_LATE && L >= G ? 1 : 0;
  }
  // 0: position pos is item (tile, is); 1: pos is the second half of a heavy
  // item (nothing to do); 2: no item at pos or later in this group.
  __device__ int map(const TcTail& q, int pos, int& tile, int& is) const {
    if (nh == 0) {
      tile = pos / q.ipt;
      is = pos - tile * q.ipt;
      return 0;
    }
    const int k = pos / G, g = pos - k * G, kh = k - h0;  // k: pass of the round robin; kh: among the heavy passes
    const int occ = kh < 0 ? 0 : (kh < 2 * hr ? G : (kh < 2 * hr + 2 ? hrem : 0));  // heavy groups of pass k
    if (g < occ) {
      if (kh & 1) return 1;
      const int j = (kh >> 1) * G + g;
      tile = j / nh;
      is = q.slot_order[j - tile * nh];
      return 0;
    }
    const int before = G * min(max(kh, 0), 2 * hr) + hrem * min(max(kh - 2 * hr, 0), 2) + min(g, occ);
    const int j = pos - before;  // light item index
    if (j >= L) return 2;
    tile = j / nl;
    is = q.slot_order[nh + j - tile * nl];
    return 0;
  }
};

// x / y rows of tile rows 4*lane .. 4*lane+3 of a gathered tile; -1 for rows
// past the tile or with a permutation entry outside [0, n) (zero-filled,
// never stored).
__device__ __forceinline__ void tile_rows4(const TcTail& q, const TcTile& t, int lane, int (&rr)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    const int r = i < t.tlen ? q.perm[t.t0 + i] : -1;
    rr[j] = (r >= 0 && r < q.n_tokens) ? r : -1;
  }
}

// Gathered rows 4*lane .. 4*lane+3 of a [128][64] bf16 tile (128 B rows, 128 B
// swizzle: 16-byte chunk c of row m at chunk c ^ (m & 7)): columns [c0, c0+64)
// of the given rows of a [n][ld] matrix of `width` columns, by 16-byte
// cp.async copies; chunks past `width` and rows of -1 are zero-filled.  Then
// this lane's arrival on `bar` once its copies have landed.
__device__ __forceinline__ void gather_rows_cp_async(uint8_t* tile, const uint16_t* base, int64_t ld, int width,
                                                     int c0, const int (&rr)[4], int lane, uint64_t* bar) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int m = 4 * lane + j;
    const uint32_t drow = smem_u32(tile) + static_cast<uint32_t>(m) * 128;
    const uint16_t* srow = base + static_cast<int64_t>(rr[j] >= 0 ? rr[j] : 0) * ld + c0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const bool ok = rr[j] >= 0 && c0 + c * 8 < width;
      cp_async16(drow + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(m) & 7u)) << 4), ok ? srow + c * 8 : base,
                 ok ? 16u : 0u);
    }
  }
  cp_async_mbar_arrive(bar);
}

// This warp's 32 TMEM lanes x N 32-bit columns from registers (column c of
// lane l: r[c] of lane l).
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] . B[smem], issued by one thread: A is M rows (TMEM
// lanes) x K bf16, two consecutive K elements per 32-bit column (the lower
// K index in the lower half).
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// Bounded wait by lane 0, result broadcast to the warp; a time-out sets the
// error flag and the CTA-wide abort flag.
template <typename SM>
__device__ __forceinline__ bool warp_wait(SM& sm, uint64_t* bar, uint32_t parity, int lane) {
  bool ok = true;
  if (lane == 0) {
    ok = mbar_wait(bar, parity, kTcWaitNs);
    if (!ok) {
      set_err(sm.t.err_flag, LORA_ERR_TIMEOUT);
      atomicExch(&sm.abort, 1);
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int R, bool CL, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) sgmv_tc_kernel(const __grid_constant__ TcParams p) {
  using Cfg = TcCfg<R>;
  using SM = TcSmem<R, CL>;
  constexpr int RP = Cfg::RP;
  constexpr int kSh = SM::kSh, kEx = SM::kEx;
  constexpr bool kHasShrink = (MODE & kModeShrink) != 0;
  constexpr bool kHasExpand = (MODE & kModeExpand) != 0;
  static_assert(!CL || MODE == kModeFused, "the cluster split serves the fused mode");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  auto& sm = *reinterpret_cast<SM*>(smem_raw);
  const TcTail& q = sm.t;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // cluster split: the C CTAs of a cluster take the same items; CTA `crank`
  // runs k-blocks [kb0, kb1) of the shrink and column blocks [b0, b1) of the
  // item's chunk, and the partial v are summed across the cluster.
  const int C = CL ? p.t.csplit : 1;
  const int crank = CL ? static_cast<int>(blockIdx.x) % C : 0;
  const int group = static_cast<int>(blockIdx.x) / C, ngroups = static_cast<int>(gridDim.x) / C;
  auto split = [&](int n, int& lo, int& hi) {
    const int per = (n + C - 1) / C;
    lo = min(n, crank * per);
    hi = min(n, lo + per);
  };
  // the k-blocks of item slot `is`: the cluster's share, or (shrink mode
  // with k-parts) the part the slot's chunk index names
  auto krange = [&](int n, int is, int& lo, int& hi) {
    if (!kHasExpand && sm.t.kparts > 1) {
      const int per = (n + sm.t.kparts - 1) / sm.t.kparts;
      lo = min(n, sm.t.item_chunk[is] * per);
      hi = min(n, lo + per);
    } else {
      split(n, lo, hi);
    }
  };

  {
    static_assert(sizeof(TcTail) % 4 == 0, "tail size");
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&p.t);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.t);
    for (int i = tid; i < static_cast<int>(sizeof(TcTail) / 4); i += kTcThreads) dst[i] = src[i];
  }
  if (warp == 4 && lane < kMaxProj) {
    prefetch_tmap(&p.tmX[lane]);
    if (LSG_TC_GATHER4_X) prefetch_tmap(&p.tmXg[lane]);
    prefetch_tmap(&p.tmA[lane]);
  }
  if (warp == 5 && lane < kMaxProj) {
    prefetch_tmap(&p.tmB[lane]);
    prefetch_tmap(&p.tmYl[lane]);
    prefetch_tmap(&p.tmYg[lane]);
    prefetch_tmap(&p.tmYs[lane]);
  }
  if constexpr (R < RP) {
    // rank 8: the v operand's columns 8..15 and the B tiles' rows 8..15 stay
    // zero (no copy or store writes them)
    if (!TcSmem<R, CL>::kVopT)
      for (int i = tid; i < 2 * Cfg::kVop / 16; i += kTcThreads)
        reinterpret_cast<uint4*>(&sm.vop[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int s = 0; s < kEx; ++s)
      for (int i = tid; i < (Cfg::kExB - Cfg::kExBCopy) / 16; i += kTcThreads)
        reinterpret_cast<uint4*>(sm.ex[s] + Cfg::kExY + Cfg::kExBCopy)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // read by the tensor cores through the async proxy
  }
  if (tid == 0) {
    for (int s = 0; s < kSh; ++s) {
      mbar_init(&sm.sh_full[s], 1);
      mbar_init(&sm.sh_empty[s], 1);
    }
    for (int s = 0; s < kEx; ++s) {
      mbar_init(&sm.ex_full[s], 1);
      mbar_init(&sm.ey_full[s], 1);
      mbar_init(&sm.ex_empty[s], 4);  // each epilogue warp, once its y stores have read the slot
    }
    mbar_init(&sm.v_full, 1);
    mbar_init(&sm.v_read, 4);
    mbar_init(&sm.vop_ready, CL ? 1 : 4);  // cluster: one local arrival + the gathered bytes
    mbar_init(&sm.rs_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 8);  // both epilogue groups' warps
      mbar_init(&sm.drain[b], 1);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 6) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // our mbarriers exist before any peer pushes into this CTA
  if (CL) cluster_arrive_relaxed();
  const uint32_t tmem = sm.tmem_base;
  pdl_launch_dependents();
  pdl_wait();
  if (CL) cluster_wait_acquire();
  // the operand swizzle below is computed on absolute shared addresses
  const bool aligned = (smem_u32(sm.sh) & 1023u) == 0;
  if (!aligned && tid == 0) set_err(q.err_flag, LORA_ERR_UNSUPPORTED);

  if (aligned && kHasShrink && warp == 4) {
    // ============================== shrink producer
    int slot = 0;
    uint32_t ph = 0, filled = 0, fill_par = 0;
    TcCursor cur;
    cur.init(q, lane);
    const TcSched sc(q, cur, lane, ngroups);
    for (int pos = group;; pos += ngroups) {
      int tile, is;
      const int step = sc.map(q, pos, tile, is);
      if (step == 2) break;
      if (step == 1) continue;
      TcTile t;
      if (!cur.find(q, lane, tile, t)) break;
      if (t.a < 0 || t.a >= q.n_slabs) continue;
      const int pj = q.item_proj[is];
      int kb0, kb1;
      krange((q.proj[pj].h_in + 63) >> 6, is, kb0, kb1);
      int rr[4] = {0, 0, 0, 0};
      if (t.row < 0) tile_rows4(q, t, lane, rr);
      bool ok = true;
      for (int kb = kb0; kb < kb1 && ok; ++kb) {
        ok = warp_wait(sm, &sm.sh_empty[slot], ph ^ 1u, lane);
        if (!ok) break;
        uint8_t* st = sm.sh[slot];
        // gathered rows: every lane copies its four rows and arrives (before
        // the producer's own arrival, so the phase waits for them)
        if (t.row < 0 && !LSG_TC_GATHER4_X)
          gather_rows_cp_async(st, q.proj[pj].x, q.proj[pj].ldx, q.proj[pj].h_in, kb * 64, rr, lane, &sm.sh_full[slot]);
        __syncwarp();
        if (LSG_TC_GATHER4_X && t.row < 0) {
          // every byte of the stage arrives by tensor copies (rows past the
          // tile read as zeros): expected before any is issued
          if (lane == 0) mbar_arrive_expect_tx(&sm.sh_full[slot], 16384u + Cfg::kShA);
          __syncwarp();
          // rows of -1 (none) read past the tensor's last row: zeros
          const int nr = q.n_tokens;
          tma_gather4(st + lane * 512, &p.tmXg[pj], kb * 64, rr[0] < 0 ? nr : rr[0], rr[1] < 0 ? nr : rr[1],
                      rr[2] < 0 ? nr : rr[2], rr[3] < 0 ? nr : rr[3], &sm.sh_full[slot]);
          if (lane == 0) tma_load_3d(st + 16384, &p.tmA[pj], 0, kb * 64, t.a, &sm.sh_full[slot]);
        } else if (lane == 0) {
          mbar_arrive_expect_tx(&sm.sh_full[slot], (t.row >= 0 ? 16384u : 0u) + Cfg::kShA);
          if (t.row >= 0) tma_load_2d(st, &p.tmX[pj], kb * 64, t.row, &sm.sh_full[slot]);
          tma_load_3d(st + 16384, &p.tmA[pj], 0, kb * 64, t.a, &sm.sh_full[slot]);
        }
        __syncwarp();
        filled |= 1u << slot;
        fill_par = (fill_par & ~(1u << slot)) | (ph << slot);
        if (++slot == kSh) {
          slot = 0;
          ph ^= 1u;
        }
      }
      if (!ok || sm.abort) break;
    }
    if (lane == 0 && sm.abort)  // no copy issued here may still be landing when the CTA leaves
      for (int s2 = 0; s2 < kSh; ++s2)
        if (filled & (1u << s2)) (void)mbar_wait(&sm.sh_full[s2], (fill_par >> s2) & 1u, kTcWaitNs);
  } else if (aligned && kHasExpand && warp == 5) {
    // ============================== expand producer
    int slot = 0;
    uint32_t ph = 0, filled = 0, fill_par = 0;
    TcCursor cur;
    cur.init(q, lane);
    const TcSched sc(q, cur, lane, ngroups);
    for (int pos = group;; pos += ngroups) {
      int tile, is;
      const int step = sc.map(q, pos, tile, is);
      if (step == 2) break;
      if (step == 1) continue;
      TcTile t;
      if (!cur.find(q, lane, tile, t)) break;
      if (t.a < 0 || t.a >= q.n_slabs) continue;
      const int pj = q.item_proj[is], ch = q.item_chunk[is];
      const TcProj& pr = q.proj[pj];
      const int c0 = ch * pr.chunk;
      int b0, b1;
      split((min(pr.chunk, pr.h_out - c0) + kBN - 1) / kBN, b0, b1);
      int rr[4] = {0, 0, 0, 0};
      if (t.row < 0) tile_rows4(q, t, lane, rr);
      bool ok = true;
      for (int b = b0; b < b1 && ok; ++b) {
        ok = warp_wait(sm, &sm.ex_empty[slot], ph ^ 1u, lane);
        if (!ok) break;
        uint8_t* st = sm.ex[slot];
        const int c = c0 + b * kBN;
        static_assert(kBH == 1, "one 64-column half per block");
        // B first, on its own barrier: the MMAs need only B, and the epilogue
        // waits for the y tile (ey_full) while they run
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.ex_full[slot], static_cast<uint32_t>(Cfg::kExBCopy));
          tma_load_2d(st + Cfg::kExY, &p.tmB[pj], c, t.a * q.rmax, &sm.ex_full[slot]);
        }
        if (t.row >= 0) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&sm.ey_full[slot], static_cast<uint32_t>(Cfg::kExY));
            tma_load_2d(st, &p.tmYl[pj], c, t.row, &sm.ey_full[slot]);
          }
        } else if (LSG_TC_GATHER4_Y) {
          // every y byte arrives by tensor gathers (rows of -1 read past the
          // tensor's last row: zeros), expected before any is issued
          if (lane == 0) mbar_arrive_expect_tx(&sm.ey_full[slot], static_cast<uint32_t>(Cfg::kExY));
          __syncwarp();
          const int nr = q.n_tokens;
          tma_gather4(st + lane * 512, &p.tmYg[pj], c, rr[0] < 0 ? nr : rr[0], rr[1] < 0 ? nr : rr[1],
                      rr[2] < 0 ? nr : rr[2], rr[3] < 0 ? nr : rr[3], &sm.ey_full[slot]);
        } else {
          // gathered rows by every lane (their arrivals), then the producer's own
          gather_rows_cp_async(st, pr.y, pr.ldy, pr.h_out, c, rr, lane, &sm.ey_full[slot]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.ey_full[slot]);
        }
        __syncwarp();
        filled |= 1u << slot;
        fill_par = (fill_par & ~(1u << slot)) | (ph << slot);
        if (++slot == kEx) {
          slot = 0;
          ph ^= 1u;
        }
      }
      if (!ok || sm.abort) break;
    }
    if (lane == 0 && sm.abort)  // no copy issued here may still be landing when the CTA leaves
      for (int s2 = 0; s2 < kEx; ++s2)
        if (filled & (1u << s2)) {
          (void)mbar_wait(&sm.ex_full[s2], (fill_par >> s2) & 1u, kTcWaitNs);
          (void)mbar_wait(&sm.ey_full[s2], (fill_par >> s2) & 1u, kTcWaitNs);
        }
  } else if (aligned && kHasShrink && warp == 6) {
    // ============================== shrink MMA issuer: v = x . A (this CTA's k-blocks)
    constexpr uint32_t kIdSh = umma_idesc_bf16(128, RP, 0, 1);
    int sslot = 0, it = 0;
    uint32_t sph = 0;
    TcCursor cur;
    cur.init(q, lane);
    const TcSched sc(q, cur, lane, ngroups);
    for (int pos = group;; pos += ngroups) {
      int tile, is;
      const int step = sc.map(q, pos, tile, is);
      if (step == 2) break;
      if (step == 1) continue;
      TcTile t;
      if (!cur.find(q, lane, tile, t)) break;
      if (t.a < 0 || t.a >= q.n_slabs) continue;
      const TcProj& pr = q.proj[q.item_proj[is]];
      int kb0, kb1;
      krange((pr.h_in + 63) >> 6, is, kb0, kb1);
      // the epilogue has read the previous item's v out of TMEM
      bool ok = it == 0 || warp_wait(sm, &sm.v_read, (it - 1) & 1, lane);
      if (!ok) break;
      tc_fence_after();
      for (int kb = kb0; kb < kb1 && ok; ++kb) {
        ok = warp_wait(sm, &sm.sh_full[sslot], sph, lane);
        if (!ok) break;
        if (t.row < 0) fence_proxy_async_smem();  // gathered x rows were written by cp.async (generic proxy)
        tc_fence_after();
        if (lane == 0) {
          const uint32_t xs = smem_u32(sm.sh[sslot]), as = xs + 16384;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = umma_desc(xs + k * 32, 16, 1024, 2);
            // A tile [64][r] MN-major: r >= 16 swizzled to 2r bytes (SBO: next 8 k-rows);
            // r = 8 without swizzle, 8x16-byte core matrices: LBO = next 8 k-rows (128 B),
            // SBO = the 8 columns past the tile (another 1 KB of this stage; results unused)
            const uint64_t bd = R >= 16 ? umma_desc(as + k * 16 * R * 2, Cfg::kShA, 8 * R * 2, umma_layout(R * 2))
                                        : umma_desc(as + k * 16 * R * 2, 128, 1024, 0);
            umma_bf16(tmem + kTmemV, ad, bd, kIdSh, kb > kb0 || k > 0);
          }
          umma_commit(&sm.sh_empty[sslot]);  // the stage is free once these MMAs have read it
        }
        __syncwarp();
        if (++sslot == kSh) {
          sslot = 0;
          sph ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) umma_commit(&sm.v_full);
      __syncwarp();
      if (sm.abort) break;
      ++it;
    }
    // every MMA issued here has completed before TMEM is released
    if (lane == 0) {
      umma_commit(&sm.drain[0]);
      (void)mbar_wait(&sm.drain[0], 0, kTcWaitNs);
    }
    __syncwarp();
  } else if (aligned && kHasExpand && warp == 7) {
    // ============================== expand MMA issuer: acc = v_hi . B + v_lo . B
    constexpr uint32_t kIdEx = umma_idesc_bf16(128, kBN, 0, 1);
    int xslot = 0, ae = 0, it = 0;
    uint32_t xph = 0;
    TcCursor cur;
    cur.init(q, lane);
    const TcSched sc(q, cur, lane, ngroups);
    for (int pos = group;; pos += ngroups) {
      int tile, is;
      const int step = sc.map(q, pos, tile, is);
      if (step == 2) break;
      if (step == 1) continue;
      TcTile t;
      if (!cur.find(q, lane, tile, t)) break;
      if (t.a < 0 || t.a >= q.n_slabs) continue;
      const TcProj& pr = q.proj[q.item_proj[is]];
      const int c0 = q.item_chunk[is] * pr.chunk;
      int b0, b1;
      split((min(pr.chunk, pr.h_out - c0) + kBN - 1) / kBN, b0, b1);
      bool ok = true;
      if (b0 < b1) {
        // (an item without blocks here is not waited for: the epilogue waits
        // for its operand itself, so this wait never falls two phases behind)
        ok = warp_wait(sm, &sm.vop_ready, it & 1, lane);
        if (!ok) break;
        if (CL) fence_proxy_async_smem();  // operand rows written by st.async, read by the tensor core
        tc_fence_after();
      }
      for (int b = b0; b < b1 && ok; ++b) {
        const int buf = ae & 1;
        ok = warp_wait(sm, &sm.acc_empty[buf], ((ae >> 1) & 1) ^ 1u, lane) &&
             warp_wait(sm, &sm.ex_full[xslot], xph, lane);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t bs = smem_u32(sm.ex[xslot]) + Cfg::kExY;
#pragma unroll
          for (int k = 0; k < RP / 16; ++k) {
            const uint64_t bd = umma_desc(bs + k * 16 * 128, RP * 128, 1024, 2);
#pragma unroll
            for (int hl = 0; hl < 2; ++hl) {
              if constexpr (TcSmem<R, CL>::kVopT) {
                // the pair in TMEM: 8 columns (16 bf16) per k-step
                umma_bf16_ta(tmem + kTmemAcc + buf * kBN, tmem + kTmemVop + hl * (RP / 2) + k * 8, bd, kIdEx,
                             k > 0 || hl > 0);
              } else {
                const uint64_t ad = umma_desc(smem_u32(sm.vop[hl]) + k * 32, 16, 8 * RP * 2, umma_layout(RP * 2));
                umma_bf16(tmem + kTmemAcc + buf * kBN, ad, bd, kIdEx, k > 0 || hl > 0);
              }
            }
          }
          if (!(withhold(3) && ae == 0)) umma_commit(&sm.acc_full[buf]);
        }
        __syncwarp();
        ++ae;
        if (++xslot == kEx) {
          xslot = 0;
          xph ^= 1u;
        }
      }
      if (!ok || sm.abort) break;
      ++it;
    }
    // every MMA issued here has completed before TMEM is released
    if (lane == 0) {
      umma_commit(&sm.drain[1]);
      (void)mbar_wait(&sm.drain[1], 0, kTcWaitNs);
    }
    __syncwarp();
  } else if (aligned && (warp < 4 || (kHasExpand && warp >= 8))) {
    // ============================== epilogue (row m = TMEM lane m): two groups
    // of four warps (0-3, 8-11); group eg turns v into the operand (group 0)
    // and updates columns [32 eg, 32 eg + 32) of every 64-column block
    const int eg = warp >> 3, wq = warp & 3;
    const int m = wq * 32 + lane;
    const uint32_t tq = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    int xslot = 0, ae = 0, it = 0;
    uint32_t xph = 0;
    int pend = -1;  // ring slot whose y stores may still be reading it
    TcCursor cur;
    cur.init(q, lane);
    // one 16-byte chunk (8 ranks) of a row as the hi / lo operand words
    auto split_hl = [](const float (&f)[8], uint32_t (&hi)[4], uint32_t (&lo)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(f[2 * e] - hf.x, f[2 * e + 1] - hf.y);
        hi[e] = *reinterpret_cast<const uint32_t*>(&h);
        lo[e] = *reinterpret_cast<const uint32_t*>(&l);
      }
    };
    // row m of the operand pair (K-major, RP-wide rows, swizzled); chunks past r keep their zeros
    auto put_operand_row = [&](const uint32_t (&v)[RP]) {
      const uint32_t hrow = smem_u32(sm.vop[0]) + static_cast<uint32_t>(m) * (RP * 2);
      const uint32_t lrow = smem_u32(sm.vop[1]) + static_cast<uint32_t>(m) * (RP * 2);
#pragma unroll
      for (int j = 0; j < R / 8; ++j) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[j * 8 + e]);
        uint32_t hi[4], lo[4];
        split_hl(f, hi, lo);
        const uint32_t ha = swz<Cfg::kSwM>(hrow + j * 16), la = swz<Cfg::kSwM>(lrow + j * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ha), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                     "r"(hi[3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(la), "r"(lo[0]), "r"(lo[1]), "r"(lo[2]),
                     "r"(lo[3])
                     : "memory");
      }
    };
    const TcSched sc(q, cur, lane, ngroups);
    for (int pos = group;; pos += ngroups) {
      int tile, is;
      const int step = sc.map(q, pos, tile, is);
      if (step == 2) break;
      if (step == 1) continue;
      TcTile t;
      if (!cur.find(q, lane, tile, t)) break;
      if (t.a < 0 || t.a >= q.n_slabs) {
        if (tid == 0 && crank == 0) set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
        continue;
      }
      const int pj = q.item_proj[is], ch = q.item_chunk[is];
      const TcProj& pr = q.proj[pj];
      const float scale = pr.scale;
      // this thread's token row (-1: none, or a corrupt permutation entry: skipped and flagged)
      int yrow = -1;
      if (m < t.tlen) {
        yrow = t.row >= 0 ? t.row + m : q.perm[t.t0 + m];
        if (yrow < 0 || yrow >= q.n_tokens) {
          if (eg == 0 && ch == 0 && crank == 0) set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
          yrow = -1;
        }
      }
      int kb0 = 0, kb1 = 0;
      if (kHasShrink) krange((pr.h_in + 63) >> 6, is, kb0, kb1);
      bool ok = true;
      if (eg == 0) {
        uint32_t v[RP];
        if constexpr (kHasShrink) {
          // ---- v (fp32, TMEM)
          ok = warp_wait(sm, &sm.v_full, it & 1, lane);
          if (!ok) break;
          tc_fence_after();
          if (kb0 < kb1) {
            if constexpr (RP == 16) {
              tmem_ld16(tq + kTmemV, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int c = 0; c < RP / 32; ++c) {
                uint32_t r32[32];
                tmem_ld32(tq + kTmemV + c * 32, r32);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[c * 32 + i] = r32[i];
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < RP; ++i) v[i] = 0u;  // no k-blocks here: a zero partial
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.v_read);  // TMEM v may take the next item's shrink
        } else {
          // ---- v from device memory (expand mode), fp32 rows in token order
#pragma unroll
          for (int i = 0; i < RP; ++i) v[i] = 0u;
          if (yrow >= 0) {
            const float4* src = reinterpret_cast<const float4*>(q.v_in + static_cast<int64_t>(yrow) * R);
#pragma unroll
            for (int j = 0; j < R / 4; ++j) {
              const float4 u = src[j];
              v[4 * j] = __float_as_uint(u.x);
              v[4 * j + 1] = __float_as_uint(u.y);
              v[4 * j + 2] = __float_as_uint(u.z);
              v[4 * j + 3] = __float_as_uint(u.w);
            }
          }
        }
        if constexpr (!kHasExpand) {
          // ---- shrink mode: v rows to device memory (fp32, token order)
          if (yrow >= 0) {
            float4* dst = reinterpret_cast<float4*>(
                q.v_out + (static_cast<int64_t>(q.kparts > 1 ? ch : 0) * q.n_tokens + yrow) * R);
#pragma unroll
            for (int j = 0; j < R / 4; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
          ++it;
          continue;
        } else if constexpr (!CL && TcSmem<R, CL>::kVopT) {
          // ---- v -> bf16 hi / lo pairs in this lane's TMEM row (the expand's A
          // operand); ranks past r are zero (the shrink's N = 16 columns past
          // rank 8 hold products that are never used)
          uint32_t hw[RP / 2], lw[RP / 2];
#pragma unroll
          for (int j = 0; j < RP / 2; ++j) {
            const float f0 = 2 * j < R ? __uint_as_float(v[2 * j]) : 0.f;
            const float f1 = 2 * j + 1 < R ? __uint_as_float(v[2 * j + 1]) : 0.f;
            const __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
            const float2 hf = __bfloat1622float2(h);
            const __nv_bfloat162 l = __floats2bfloat162_rn(f0 - hf.x, f1 - hf.y);
            hw[j] = *reinterpret_cast<const uint32_t*>(&h);
            lw[j] = *reinterpret_cast<const uint32_t*>(&l);
          }
          tmem_st<RP / 2>(tq + kTmemVop, hw);
          tmem_st<RP / 2>(tq + kTmemVop + RP / 2, lw);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.vop_ready);
        } else if constexpr (!CL) {
          // ---- v -> bf16 operands hi, lo (K-major, 2*RP-byte swizzle)
          put_operand_row(v);
          fence_proxy_async_smem();  // the tensor core reads the operands through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.vop_ready);
        } else {
          // ---- reduce-scatter: row m's partial to the CTA that owns the row
          const int rpo = 128 / C;  // rows per owner
          const int own = m / rpo, ml = m - own * rpo;
          if (tid == 0) {
            mbar_arrive_expect_tx(&sm.rs_full, 128u * R * 4u);    // C ranks x rpo rows x r fp32
            mbar_arrive_expect_tx(&sm.vop_ready, 128u * R * 4u);  // 128 rows x r x (hi + lo) bf16
          }
          {
            const uint32_t dst = mapa_shared(smem_u32(&sm.rbuf[(crank * rpo + ml) * R]), own);
            const uint32_t bar = mapa_shared(smem_u32(&sm.rs_full), own);
#pragma unroll
            for (int j = 0; j < R / 4; ++j)
              st_async_v4(dst + j * 16,
                          make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                      __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])),
                          bar);
          }
          ok = warp_wait(sm, &sm.rs_full, it & 1, lane);
          if (!ok) break;
          // ---- sum the C partials of the owned rows (fixed order: the same v in
          // every CTA), split into hi / lo and all-gather into every CTA's operand
          for (int w = tid; w < rpo * (R / 8); w += kTcEpiThreads) {
            const int lr = w / (R / 8), j = w - lr * (R / 8);
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 0.f;
            for (int src = 0; src < C; ++src) {
              const float4* pp = reinterpret_cast<const float4*>(&sm.rbuf[(src * rpo + lr) * R + j * 8]);
              const float4 u0 = pp[0], u1 = pp[1];
              f[0] += u0.x;
              f[1] += u0.y;
              f[2] += u0.z;
              f[3] += u0.w;
              f[4] += u1.x;
              f[5] += u1.y;
              f[6] += u1.z;
              f[7] += u1.w;
            }
            uint32_t hi[4], lo[4];
            split_hl(f, hi, lo);
            const uint32_t mrow = static_cast<uint32_t>(crank * rpo + lr) * (RP * 2) + j * 16;
            const uint32_t ha = swz<Cfg::kSwM>(smem_u32(sm.vop[0]) + mrow);
            const uint32_t la = swz<Cfg::kSwM>(smem_u32(sm.vop[1]) + mrow);
            const uint32_t bar = smem_u32(&sm.vop_ready);
            for (int d = 0; d < C; ++d) {
              const uint32_t rb = mapa_shared(bar, d);
              st_async_u4(mapa_shared(ha, d), hi[0], hi[1], hi[2], hi[3], rb);
              st_async_u4(mapa_shared(la, d), lo[0], lo[1], lo[2], lo[3], rb);
            }
          }
          // the whole operand is here before the next item's expectations are
          // registered (and the expand MMAs of this item may start)
          ok = warp_wait(sm, &sm.vop_ready, it & 1, lane);
          if (!ok) break;
        }
      }  // eg == 0
      if constexpr (kHasExpand) {
        // ---- expand blocks: y = bf16(y + s * acc)
        const int c0 = ch * pr.chunk;
        int b0, b1;
        split((min(pr.chunk, pr.h_out - c0) + kBN - 1) / kBN, b0, b1);
        const bool contig = t.row >= 0;
        const int full_rows = contig ? (t.tlen >> 5) << 5 : 0;  // rows stored by TMA boxes
        // gathered tile: rows in a group of four valid rows go out by one
        // four-row scatter (lane j of the quarter's warp: rows 4j .. 4j+3)
        const unsigned vmask = __ballot_sync(0xffffffffu, yrow >= 0);
        const bool by_tensor_store =
            contig ? m < full_rows : (LSG_TC_SCATTER4 && ((vmask >> (lane & ~3)) & 0xFu) == 0xFu);
        int yr4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) yr4[k] = __shfl_sync(0xffffffffu, yrow, (4 * lane + k) & 31);
        const bool scatter_lane = LSG_TC_SCATTER4 && !contig && lane < 8 && ((vmask >> (4 * lane)) & 0xFu) == 0xFu;
        for (int b = b0; b < b1 && ok; ++b) {
          const int buf = ae & 1;
          ok = warp_wait(sm, &sm.acc_full[buf], (ae >> 1) & 1, lane) && warp_wait(sm, &sm.ey_full[xslot], xph, lane);
          if (!ok) break;
          tc_fence_after();
          uint8_t* st = sm.ex[xslot];
          const int c = c0 + b * kBN;
          {
            // this group's 32 columns of the block
            uint32_t acc[32];
            tmem_ld32(tq + kTmemAcc + buf * kBN + eg * 32, acc);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);  // accumulator in registers: TMEM buffer free
            const uint32_t rbase = smem_u32(st) + static_cast<uint32_t>(m) * 128;
            uint16_t* yp = yrow >= 0 ? pr.y + static_cast<int64_t>(yrow) * pr.ldy : nullptr;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = eg * 4 + i;  // 16-byte chunk of the 64-column block
              const uint32_t addr = rbase + ((static_cast<uint32_t>(j) ^ (m & 7u)) << 4);
              uint32_t yw[4];
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(yw[0]), "=r"(yw[1]), "=r"(yw[2]), "=r"(yw[3])
                           : "r"(addr));
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&yw[e]));
                const __nv_bfloat162 o =
                    __floats2bfloat162_rn(yf.x + scale * __uint_as_float(acc[i * 8 + 2 * e]),
                                          yf.y + scale * __uint_as_float(acc[i * 8 + 2 * e + 1]));
                yw[e] = *reinterpret_cast<const uint32_t*>(&o);
              }
              if (by_tensor_store) {
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(yw[0]), "r"(yw[1]),
                             "r"(yw[2]), "r"(yw[3])
                             : "memory");
              } else if (yp != nullptr && c + j * 8 < pr.h_out) {
                // rows past the last whole group of 32 (contiguous tile) or of
                // four (gathered tile): written directly (16-byte stores)
                *reinterpret_cast<uint4*>(yp + c + j * 8) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
              }
            }
          }
          fence_proxy_async_smem();  // our y updates, visible to the tensor stores
          named_bar_sync(3 + wq, 64);  // the two warps of this lane quarter are done with the block
          if (eg == 0) {
            // each lane quarter stores its own 32 rows: one 64-column box, or
            // four-row scatters of a gathered tile
            const int g = wq * 32;
            if (lane == 0 && g + 32 <= full_rows && c < pr.h_out) tma_store_2d(&p.tmYs[pj], c, t.row + g, st + g * 128);
            if (scatter_lane && c < pr.h_out)
              tma_scatter4(&p.tmYg[pj], c, yr4[0], yr4[1], yr4[2], yr4[3], st + (g + 4 * lane) * 128);
            bulk_commit();
            if (LSG_TC_RELEASE_EARLY) {
              bulk_wait_read0();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.ex_empty[xslot]);  // y rows read by the stores, B tile by the MMAs
            } else if (pend >= 0) {
              // the previous block's stores have read their slot (this block's may
              // still be reading): this quarter's share of that slot goes back
              bulk_wait_read1();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.ex_empty[pend]);  // y rows read by the stores, B tile read by the MMAs
            }
            pend = xslot;
          }
          ++ae;
          if (++xslot == kEx) {
            xslot = 0;
            xph ^= 1u;
          }
        }
      }
      if (!ok || sm.abort) break;
      ++it;
    }
  }
  if (aligned && warp < 4) bulk_wait_read0();  // the last y stores have read shared memory
  tc_fence_before();
  __syncthreads();
  if (CL) {
    // no CTA leaves while a peer may still write into its shared memory
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

namespace {

// Co-resident CTA groups of C CTAs (one CTA per SM) of a kernel instance on
// the current device (clusters of C when CL); sets the kernel's shared-memory
// attribute on first use.
template <int R, bool CL, int MODE>
lora_status tc_groups(int C, int& groups) {
  static std::mutex mu;
  static int cache[64][kMaxC + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(mu);
    groups = cache[dev & 63][C];
  }
  if (groups > 0) return LORA_OK;
  auto kern = sgmv_tc_kernel<R, CL, MODE>;
  static_assert(sizeof(TcSmem<R, CL>) <= 227 * 1024, "shared memory per CTA");
  const size_t smem = sizeof(TcSmem<R, CL>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return LORA_ERR_CUDA;
  if (CL) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute at[1];
    cfg.gridDim = dim3(C * 64);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&groups, kern, &cfg) != cudaSuccess) return LORA_ERR_CUDA;
  } else if (cudaDeviceGetAttribute(&groups, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    return LORA_ERR_CUDA;
  }
  groups = std::max(1, groups);
  std::lock_guard<std::mutex> lk(mu);
  cache[dev & 63][C] = groups;
  return LORA_OK;
}

template <int R, bool CL, int MODE>
lora_status launch_tc_rc(TcParams& prm, const SgmvCall& call, int tiles_bound, cudaStream_t stream) {
  constexpr bool kHasShrink = (MODE & kModeShrink) != 0;
  constexpr bool kHasExpand = (MODE & kModeExpand) != 0;
  auto kern = sgmv_tc_kernel<R, CL, MODE>;
  static_assert(sizeof(TcSmem<R, CL>) <= 227 * 1024, "shared memory per CTA");
  const size_t smem = sizeof(TcSmem<R, CL>);
  const int C = prm.t.csplit;
  const uint64_t n = static_cast<uint64_t>(call.seg.n_tokens);
  for (int i = 0; i < call.n_proj; ++i) {
    const ProjArgs& a = call.proj[i];
    lora_status s;
    if (kHasShrink) {
      const uint64_t dims[2] = {static_cast<uint64_t>(a.h_in), n};
      const uint64_t str[1] = {static_cast<uint64_t>(a.ldx) * 2};
      const uint32_t box[2] = {64, 128};
      if ((s = encode_tmap_bf16(&prm.tmX[i], a.x, 2, dims, str, box, 128)) != LORA_OK) return s;
      if (LSG_TC_GATHER4_X) {
        const uint32_t box_g[2] = {64, 1};
        if ((s = encode_tmap_bf16(&prm.tmXg[i], a.x, 2, dims, str, box_g, 128)) != LORA_OK) return s;
      }
      const uint64_t adims[3] = {static_cast<uint64_t>(R), static_cast<uint64_t>(a.h_in),
                                 static_cast<uint64_t>(prm.t.n_slabs)};
      const uint64_t astr[2] = {static_cast<uint64_t>(R) * 2, static_cast<uint64_t>(a.h_in) * prm.t.rmax * 2};
      const uint32_t abox[3] = {static_cast<uint32_t>(R), 64, 1};
      if ((s = encode_tmap_bf16(&prm.tmA[i], a.A, 3, adims, astr, abox, R >= 16 ? R * 2 : 0)) != LORA_OK) return s;
    }
    if (kHasExpand) {
      const uint64_t bdims[2] = {static_cast<uint64_t>(a.h_out), static_cast<uint64_t>(prm.t.n_slabs) * prm.t.rmax};
      const uint64_t bstr[1] = {static_cast<uint64_t>(a.h_out) * 2};
      const uint32_t bbox[2] = {64, static_cast<uint32_t>(R)};
      if ((s = encode_tmap_bf16(&prm.tmB[i], a.B, 2, bdims, bstr, bbox, 128)) != LORA_OK) return s;
      const uint64_t dims[2] = {static_cast<uint64_t>(a.h_out), n};
      const uint64_t str[1] = {static_cast<uint64_t>(a.ldy) * 2};
      const uint32_t box_l[2] = {64, 128}, box_g[2] = {64, 1}, box_s[2] = {64, 32};
      if ((s = encode_tmap_bf16(&prm.tmYl[i], a.y, 2, dims, str, box_l, 128)) != LORA_OK) return s;
      if ((s = encode_tmap_bf16(&prm.tmYg[i], a.y, 2, dims, str, box_g, 128)) != LORA_OK) return s;
      if ((s = encode_tmap_bf16(&prm.tmYs[i], a.y, 2, dims, str, box_s, 128)) != LORA_OK) return s;
    }
  }

  int max_groups = 0;
  if (const lora_status st = tc_groups<R, CL, MODE>(C, max_groups); st != LORA_OK) return st;
  const int64_t items = static_cast<int64_t>(tiles_bound) * prm.t.ipt;
  const int groups = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(max_groups, items)));

  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute at[2];
  int na = 0;
  cfg.gridDim = dim3(groups * C);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  if (CL) {
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

// Work plan: items are (tile, projection, column chunk) taken by groups of C
// CTAs.  For each C in {1, 2, 4, 8} the columns are cut into enough chunks
// for one pass of items over the co-resident groups (at least one chunk of
// about kChunkCols columns per projection; each extra chunk re-reads the
// tile's x and the A slab for its own shrink); the plan with the fewest bytes
// per CTA over all passes wins (ties: the smaller C).  The shrink and expand
// modes run one CTA per item; the shrink mode has one item per tile.
template <int R, int MODE>
lora_status plan_and_launch(const SgmvCall& call, cudaStream_t stream) {
  constexpr bool kHasShrink = (MODE & kModeShrink) != 0;
  constexpr bool kHasExpand = (MODE & kModeExpand) != 0;
  TcParams prm{};
  const int n = call.seg.n_tokens;
  const int tiles_est = std::max(1, ceil_div(n, 128));
  int64_t cols = 0;
  int min_kb = 1 << 30;
  for (int i = 0; i < call.n_proj; ++i) {
    cols += kHasExpand ? call.proj[i].h_out : 0;
    if (kHasShrink) min_kb = std::min(min_kb, ceil_div(call.proj[i].h_in, 64));
  }
  struct Plan {
    int C = 0, nch[kMaxProj] = {}, ipt = 0;
    double cost = 0;
  } best;
  const int c_max = MODE == kModeFused ? kMaxC : 1;
  for (int C = 1; C <= c_max && C <= min_kb; C *= 2) {
    int G = 0;
    const lora_status st = C == 1 ? tc_groups<R, false, MODE>(1, G) : tc_groups<R, (MODE == kModeFused), MODE>(C, G);
    if (st != LORA_OK) return st;
    const int target = std::clamp(G / tiles_est, 1, kMaxItemsPerTile);  // items per tile
    Plan pl;
    pl.C = C;
    int base = 0;
    for (int i = 0; i < call.n_proj; ++i)
      base += kHasExpand ? std::clamp(ceil_div(call.proj[i].h_out, kChunkCols), 1, 8) : 1;
    bool ok = true;
    double bytes = 0;
    for (int i = 0; i < call.n_proj && ok; ++i) {
      const ProjArgs& a = call.proj[i];
      if (!kHasExpand) {
        pl.nch[i] = 1;
        pl.ipt += 1;
        bytes += 128.0 * a.h_in * 2 + a.h_in * R * 2;
        continue;
      }
      int nch = std::clamp(ceil_div(a.h_out, kChunkCols), 1, 8);
      if (base < target) {
        const int share = static_cast<int>((static_cast<int64_t>(target) * a.h_out + cols - 1) / cols);
        nch = std::max(nch, std::min(share, std::max(1, a.h_out / (128 * C))));
        nch = std::min(nch, kMaxItemsPerTile / call.n_proj);
      }
      const int chunk = round_up(ceil_div(a.h_out, nch), 128);
      nch = ceil_div(a.h_out, chunk);
      pl.nch[i] = nch;
      pl.ipt += nch;
      // every CTA of a cluster needs an expand block of every item
      if (ceil_div(a.h_out - (nch - 1) * chunk, kBN) < C) ok = false;
      bytes += static_cast<double>(nch) * (kHasShrink ? 128.0 * a.h_in * 2 + a.h_in * R * 2 : 128.0 * R * 4) +
               static_cast<double>(a.h_out) * (128 * 4 + R * 2);
    }
    if (!ok) continue;
    const int64_t items = static_cast<int64_t>(tiles_est) * pl.ipt;
    const int64_t rounds = (items + G - 1) / G;
    pl.cost = static_cast<double>(rounds) * bytes / pl.ipt / C;
    if (best.C == 0 || pl.cost < best.cost * 0.999) best = pl;
  }
  if (best.C == 0) return LORA_ERR_UNSUPPORTED;
  // Shrink mode into k-partial slices: a batch of few tiles splits each
  // tile's k-blocks over up to v_parts_max items, so that about one item per
  // co-resident CTA streams its part of x (one item per tile would leave most
  // SMs idle and each item a long serial stream).
  int kparts = 1;
  if constexpr (MODE == kModeShrink) {
    if (call.v_parts_max > 1) {
      int G = 0;
      const lora_status st = tc_groups<R, false, MODE>(1, G);
      if (st != LORA_OK) return st;
      kparts = std::clamp(G / (tiles_est * call.n_proj), 1,
                          std::min({call.v_parts_max, min_kb, kMaxItemsPerTile / call.n_proj}));
      for (int i = 0; i < call.n_proj; ++i) best.nch[i] = kparts;
    }
  }
  if (call.v_parts != nullptr) *call.v_parts = kparts;
  int ipt = 0;
  for (int i = 0; i < call.n_proj; ++i) {
    const ProjArgs& a = call.proj[i];
    TcProj& t = prm.t.proj[i];
    t.x = a.x;
    t.ldx = a.ldx;
    t.y = a.y;
    t.ldy = a.ldy;
    t.h_in = a.h_in;
    t.h_out = a.h_out;
    t.scale = a.scale;
    t.chunk = kHasExpand ? round_up(ceil_div(a.h_out, best.nch[i]), 128) : 0;
    for (int c = 0; c < best.nch[i]; ++c) {
      prm.t.item_proj[ipt] = static_cast<int8_t>(i);
      prm.t.item_chunk[ipt] = static_cast<int8_t>(c);
      ++ipt;
    }
  }
  // Heavy item slots: an item's time is about max(its shrink k-blocks x
  // LSG_TC_COST_KB, its expand blocks x LSG_TC_COST_BLK) (us per block
  // measured on B300; the shrink and the expand of consecutive items
  // overlap); a slot of at least 1.5x the median item weighs two positions.
  {
    double cost[kMaxItemsPerTile], sorted[kMaxItemsPerTile];
    for (int k = 0; k < ipt; ++k) {
      const ProjArgs& a = call.proj[prm.t.item_proj[k]];
      const TcProj& t = prm.t.proj[prm.t.item_proj[k]];
      const int kb = kHasShrink ? ceil_div(a.h_in, 64) : 0;
      const int cols = kHasExpand ? std::min(t.chunk, a.h_out - prm.t.item_chunk[k] * t.chunk) : 0;
      cost[k] = sorted[k] = std::max(LSG_TC_COST_KB * kb, LSG_TC_COST_BLK * ceil_div(cols, kBN));
    }
    std::sort(sorted, sorted + ipt);
    const double median = sorted[(ipt - 1) / 2];
    int nh = 0;
    for (int k = 0; k < ipt; ++k)
      if (cost[k] >= 1.5 * median) prm.t.slot_order[nh++] = static_cast<int8_t>(k);
    int nl = nh;
    for (int k = 0; k < ipt; ++k)
      if (!(cost[k] >= 1.5 * median)) prm.t.slot_order[nl++] = static_cast<int8_t>(k);
    prm.t.n_heavy = LSG_TC_HEAVY_FIRST ? nh : 0;
    if (!LSG_TC_HEAVY_FIRST)
      for (int k = 0; k < ipt; ++k) prm.t.slot_order[k] = static_cast<int8_t>(k);
  }
  prm.t.csplit = best.C;
  prm.t.kparts = kparts;
  prm.t.slot_of = call.slot_of;
  prm.t.rank_of = call.rank_of;
  prm.t.n_slabs = call.slot_of ? call.n_slots : call.n_adapters;
  prm.t.rmax = call.slot_of ? call.r_max : R;
  prm.t.rank = R;
  prm.t.perm = call.seg.perm;
  prm.t.seg_offsets = call.seg.seg_offsets;
  prm.t.seg_adapter = call.seg.seg_adapter;
  prm.t.num_segments = call.seg.num_segments;
  prm.t.err_flag = call.err_flag;
  prm.t.v_out = call.v_out;
  prm.t.v_in = call.v_in;
  prm.t.n_proj = call.n_proj;
  prm.t.ipt = ipt;
  prm.t.n_tokens = n;
  prm.t.max_segments = call.seg.max_segments;
  prm.t.n_adapters = call.n_adapters;
  // upper bound of the tiles of segments of at least kLongSeg tokens
  const int tiles_bound = ceil_div(n, 128) + n / kLongSeg;
  if constexpr (MODE == kModeFused) {
    if (best.C > 1) return launch_tc_rc<R, true, MODE>(prm, call, tiles_bound, stream);
  }
  return launch_tc_rc<R, false, MODE>(prm, call, tiles_bound, stream);
}

template <int R>
lora_status launch_mode(const SgmvCall& call, cudaStream_t stream) {
  switch (call.mode) {
    case kModeShrink: return plan_and_launch<R, kModeShrink>(call, stream);
    case kModeExpand: return plan_and_launch<R, kModeExpand>(call, stream);
    default: return plan_and_launch<R, kModeFused>(call, stream);
  }
}

}  // namespace

// Launched when segments can be long: tokens per possible segment >= 64
// (known on the host without reading the segmentation), or a batch of at
// least kTcMinTokens tokens, where one extra launch that may find no long
// segment costs little next to the step.  Segments it does not take are left
// to the split-K kernel, which handles any segment.
constexpr int kTcMinTokens = 512;
bool sgmv_tc_applicable(const SgmvCall& call) {
  const int n = call.seg.n_tokens;
  const int max_seg = std::max(1, std::min(n, call.n_adapters));
  return (call.r == 8 || call.r == 16 || call.r == 32 || call.r == 64) && n >= kLongSeg &&
         (n / max_seg >= kLongSeg || n >= kTcMinTokens);
}

lora_status launch_sgmv_tc(const SgmvCall& call, cudaStream_t stream) {
  switch (call.r) {
    case 8: return launch_mode<8>(call, stream);
    case 16: return launch_mode<16>(call, stream);
    case 32: return launch_mode<32>(call, stream);
    case 64: return launch_mode<64>(call, stream);
    default: return LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace lsg
