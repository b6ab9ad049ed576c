// The backbone projection with the LoRA delta in one output pass: SGMV's
// expand fused into the backbone GEMM, so y is written once.
//
//   y[i,:] = x[i,:] . W + s * ((x[i,:] . A[a_i]) . B[a_i])
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Summary":
// the backbone runs as one ordinary GEMM over the whole batch and the
// per-adapter low-rank additions are computed together, requests of one
// adapter grouped; "Interesting ideas" I1: the shared computation and the
// per-tenant one are split.  Here the per-tenant expand joins the shared
// GEMM's accumulator, so the LoRA path adds no y read or write of its own.
//
// A call is three launches on the stream:
//  1. the tensor-tile SGMV kernel in its shrink mode: v = x . A[a] (fp32,
//     token order, into the caller's workspace) for the tokens of segments of
//     at least kLongSeg tokens;
//  2. gemm_lora_kernel (below): for each tile of 128 tokens (in the
//     segmentation's order) x 256 output columns, acc = x . W on the tensor
//     cores (tcgen05, fp32 in TMEM), then, for each long segment that
//     overlaps the tile, acc += (s * v) . B[a] with v as a bf16 pair hi + lo
//     (16 bits of its mantissa) and its rows outside the segment zero; y =
//     bf16(acc) once.  Tokens of short segments and tokens whose adapter id
//     is invalid get y = x . W here;
//  3. the split-K SGMV kernel adds the delta of the short segments to y in
//     place (a step that finds no short segment does nothing).
//
// gemm_lora_kernel: one CTA per SM, persistent.  A unit is a pair of token
// tiles (256 tokens) x one column tile of 256: both 128 x 256 accumulators
// (all 512 TMEM columns) take their MMAs from the same W stage, so each W
// byte brought from L2 serves 256 tokens (128 flop per operand byte, against
// 85 for one tile).  Units, column tiles inner, are dealt round robin over the
// CTAs, so the units in flight together cover a few token tiles and all of W:
// both stay in L2.  Only whole waves of pairs are dealt as pairs; when the
// pairs left over fill at most half a wave they are dealt as single tiles
// (twice as many units, each about a fifth shorter than a pair), so the last
// wave is shorter.  Six warps:
//   warps 0-3  epilogue (warp w: TMEM lane quarter w; thread = tile row): the
//              operand (s v as bf16 hi + lo) of each long segment, then y
//              from the accumulators (a warp's 32 contiguous rows through a
//              swizzled staging box and one TMA store, other rows by 16-byte
//              stores)
//   warp 4     producer: TMA x tiles [128][64] (a 2-D box, one 256-row box
//              for two adjacent contiguous tiles, or four-row gathers through
//              the permutation), W tiles [64][256] (one 3-D box of four
//              [64][64] blocks, or four boxes; MN-major, 128 B swizzle), B
//              tiles [r][256]
//   warp 5     TMEM allocation; one thread issues the MMAs (M = 128, N = 256)
// The ring's stages (3 of 64 KB) hold the unit's x tiles and one W tile.
// TMEM holds no second pair of accumulators, so the issuer starts the next
// unit once the epilogue has read both.  Single-tile builds (LSG_GL_PAIR=0)
// keep two accumulators that alternate between units instead.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace lsg {

constexpr int kGlThreads = 192;
constexpr int kGlBN = 256;     // output columns per tile (MMA N)
constexpr int kGlMaxRuns = 3;  // long segments (>= 64 tokens) a 128-token window can overlap
// Build-time knob, set by measurement: units of two token tiles sharing each
// W stage (1), or of one token tile with alternating accumulators (0).
#ifndef LSG_GL_PAIR
#define LSG_GL_PAIR 1
#endif
// Fewer, larger tensor copies per stage (1): a pair of adjacent contiguous
// tiles as one 256-row x box, and W as one 3-D box of its four 64-column
// blocks when h_out is a multiple of 64; else a box per tile and per block.
#ifndef LSG_GL_WIDE
#define LSG_GL_WIDE 1
#endif
// k-partial slices the shrink launch may split each long tile into (at most
// kGlVParts), so that its items cover more SMs.  Measured on the 13B layer
// (6224 tokens, 49 tiles): at most 1 / 2 / 3 parts 3723 / 3652 / 3717 us.
#ifndef LSG_GL_SHRINK_PARTS
#define LSG_GL_SHRINK_PARTS 2
#endif
// Clusters of LSG_GL_CM CTAs (1 or 2): the CTAs of a cluster take the same
// column tile of different token tiles, each loads a 1/CM share of the W
// tile and multicasts it to every CTA of the cluster, so each SM reads
// 1/CM of the W bytes from L2.  A ring slot is refilled only after every CTA
// of the cluster has consumed it.  Measured no faster on the 13B layer (each
// SM still receives the whole stage), so CTAs run alone.
#ifndef LSG_GL_CM
#define LSG_GL_CM 1
#endif
constexpr int kGlCM = LSG_GL_CM;
static_assert(kGlCM == 1 || kGlCM == 2, "cluster size");
constexpr int kGlMT = LSG_GL_PAIR ? 2 : 1;       // token tiles per unit, at most
constexpr int kGlStages = kGlMT == 2 ? 3 : 4;    // ring stages (64 KB / 48 KB)
constexpr int kGlBufs = kGlMT == 2 ? 1 : 2;      // accumulator sets in the 512 TMEM columns
constexpr uint64_t kGlWaitNs = LSG_WAIT_LIMIT_NS;

#ifdef LSG_TEST_HOOKS
__device__ int g_test_withhold_gl;
__device__ __forceinline__ bool gl_withhold(int what) { return *(volatile int*)&g_test_withhold_gl == what; }
lora_status test_withhold_gl(int what) {
  return cuda_status(cudaMemcpyToSymbol(g_test_withhold_gl, &what, sizeof(int)));
}
#else
__device__ __forceinline__ bool gl_withhold(int) { return false; }
#endif

struct GlTail {
  const int32_t* perm;
  const int32_t* seg_offsets;
  const int32_t* seg_adapter;
  const int32_t* num_segments;
  const float* v;  // [vparts][n][r] fp32: k-partial sums of v, rows of long-segment tokens
  uint16_t* y;
  int64_t ldy;
  int64_t vslice;  // floats between the partial slices of v (n * r)
  int32_t* err_flag;
  int32_t n_tokens, max_segments, n_adapters, h_in, h_out;
  int32_t m_tiles, n_tiles, k_blocks;
  int32_t units;       // units of the launch
  int32_t pair_units;  // units [0, pair_units) take two token tiles, the rest one
  int32_t use_runs;    // long segments' expands are fused here (their v was computed)
  int32_t vparts;      // partial slices of v to sum
  int32_t w3d;         // W tiles as one 3-D box (tmW3)
  float scale;
};

struct GlParams {
  CUtensorMap tmX;   // x [n][h_in], box {64, 128}, 128 B swizzle
  CUtensorMap tmXg;  // x, box {64, 1} (four-row gathers)
  CUtensorMap tmX2;  // x, box {64, 256} (two adjacent contiguous tiles)
  CUtensorMap tmW;   // W [h_in][h_out], box {64, 64}, 128 B swizzle
  CUtensorMap tmW3;  // W as [h_out / 64][h_in][64], box {64, 64, 4}, 128 B swizzle (w3d)
  CUtensorMap tmB;   // B pool [P][r][h_out], box {64, RP, 1} (rows past r read zeros), 128 B swizzle
  CUtensorMap tmY;   // y [n][h_out], box {64, 32}, 128 B swizzle (stores of 32 contiguous rows)
  GlTail t;
};

template <int R>
struct GlCfg {
  static constexpr int RP = R < 16 ? 16 : R;  // MMA K of the expand (rank 8 padded with zero rows)
  static constexpr int kX = 16384;            // x tile [128][64]
  static constexpr int kW = 32768;            // W tile [64][256]
  static constexpr int kStage = kGlMT * kX + kW;
  static constexpr int kB = RP * 512;         // B tile [RP][256] (in the W part of a stage)
  static constexpr int kVop = 128 * RP * 2;   // one bf16 operand [128][RP]
  static constexpr int kStg = 4 * 2 * 4096;   // y staging: per epilogue warp two [32][64] bf16 boxes
  static constexpr int kOpSt = 2 * kVop > kStg ? 2 * kVop : kStg;  // operand pair, or y staging
  static constexpr uint32_t kSwM = (RP * 2) / 16 - 1;
  static_assert(kB <= kW, "B tile fits a stage");
};

template <int R>
struct GlSmem {
  alignas(1024) uint8_t st[kGlStages][GlCfg<R>::kStage];
  // the operand pair (hi at 0, lo at kVop) while a unit's long segments are
  // expanded; the epilogue's y staging after its accumulators are complete
  alignas(1024) uint8_t opst[GlCfg<R>::kOpSt];
  alignas(16) GlTail t;
  alignas(8) uint64_t full[kGlStages];
  uint64_t empty[kGlStages];
  uint64_t acc_full[kGlBufs];
  uint64_t acc_empty[kGlBufs];
  uint64_t op_full;   // the operand of the next long segment is in shared memory
  uint64_t op_empty;  // the expand MMAs of the last one completed
  uint64_t drain;     // the MMA issuer, at exit: its MMAs have completed
  uint32_t tmem_base;
  int32_t abort;
};

// A 128-token window of the segmentation's order and the long segments that
// overlap it.  Computed by a full warp (every lane gets the same result).
struct GlTile {
  int t0, tlen;
  int row;  // first x / y row when the window's rows are contiguous, else -1
  int nrun;
  int a[kGlMaxRuns], lo[kGlMaxRuns], hi[kGlMaxRuns];  // adapter, tile rows [lo, hi)
};

__device__ __forceinline__ void gl_tile(const GlTail& q, int S, int mt, int lane, GlTile& t) {
  const int n = q.n_tokens;
  t.t0 = mt * 128;
  t.tlen = min(128, n - t.t0);
  t.row = -1;
  t.nrun = 0;
  if (t.tlen <= 0) return;  // the second tile of the last pair, past the batch
  const int f = q.perm[t.t0];
  bool c = f >= 0 && f + t.tlen <= n;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    if (i < t.tlen) c &= q.perm[t.t0 + i] == f + i;
  }
  t.row = __all_sync(0xffffffffu, c) ? f : -1;
  if (!q.use_runs || S <= 0) return;
  const int n_valid = q.seg_offsets[S];
  if (t.t0 >= n_valid) return;
  // the segment holding position t0: the last s with seg_offsets[s] <= t0
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (q.seg_offsets[mid] <= t.t0) lo = mid;
    else hi = mid - 1;
  }
  for (int s = lo; s < S && t.nrun < kGlMaxRuns; ++s) {
    const int o = q.seg_offsets[s], e = q.seg_offsets[s + 1];
    if (o >= t.t0 + t.tlen) break;
    const int a = q.seg_adapter[s];
    if (e - o >= kLongSeg && a >= 0 && a < q.n_adapters && e <= n) {
      const int rlo = max(o, t.t0) - t.t0, rhi = min(e, t.t0 + t.tlen) - t.t0;
#pragma unroll
      for (int j = 0; j < kGlMaxRuns; ++j)
        if (j == t.nrun) {
          t.a[j] = a;
          t.lo[j] = rlo;
          t.hi[j] = rhi;
        }
      ++t.nrun;
    }
  }
}

// Unit u of a cluster, for its CTA `crank`: token tiles [mt, mt + ntl) x
// column tile nt.  A unit takes a group of kGlCM pairs, pair (g kGlCM + crank)
// for CTA crank.  Units below pair_units are whole pairs (2p, 2p + 1), column
// tiles inner; the units after them split the remaining groups into their
// first and second tiles, in the same order.
struct GlUnit {
  int mt, ntl, nt;
};

__device__ __forceinline__ GlUnit gl_unit(const GlTail& q, int u, int crank) {
  if (kGlMT == 1) {
    const int g = u / q.n_tiles;
    return GlUnit{g * kGlCM + crank, 1, u - g * q.n_tiles};
  }
  if (u < q.pair_units) {
    const int g = u / q.n_tiles;
    return GlUnit{2 * (g * kGlCM + crank), 2, u - g * q.n_tiles};
  }
  const int s = u - q.pair_units, w = q.pair_units + (s >> 1), g = w / q.n_tiles;
  return GlUnit{2 * (g * kGlCM + crank) + (s & 1), 1, w - g * q.n_tiles};
}

// The unit's tiles (a full warp); a tile index past the unit gets no rows.
__device__ __forceinline__ bool gl_tiles(const GlTail& q, int S, const GlUnit& un, int lane,
                                         GlTile (&t)[kGlMT]) {
  bool any = false;
#pragma unroll
  for (int mi = 0; mi < kGlMT; ++mi) {
    if (mi < un.ntl) {
      gl_tile(q, S, un.mt + mi, lane, t[mi]);
    } else {
      t[mi].tlen = 0;
      t[mi].row = -1;
      t[mi].nrun = 0;
    }
    any |= t[mi].tlen > 0;
  }
  return any;
}

// A unit seen from one CTA of its cluster (a full warp): its own tiles, and
// whether any CTA of the cluster has rows; nslot[mi]: the long segments'
// expand slots of tile mi, the most any CTA of the cluster has (a CTA with
// fewer fills the rest with empty slots, so the rings stay in step).
struct GlView {
  bool own, all;
  int nslot[kGlMT];
};

__device__ __forceinline__ GlView gl_view(const GlTail& q, int S, int u, int crank, int lane, GlTile (&t)[kGlMT]) {
  GlView v;
  v.own = gl_tiles(q, S, gl_unit(q, u, crank), lane, t);
  v.all = v.own;
#pragma unroll
  for (int mi = 0; mi < kGlMT; ++mi) v.nslot[mi] = t[mi].nrun;
#pragma unroll
  for (int k = 0; k < kGlCM; ++k) {
    if (k == crank) continue;
    GlTile tk[kGlMT];
    v.all |= gl_tiles(q, S, gl_unit(q, u, k), lane, tk);
#pragma unroll
    for (int mi = 0; mi < kGlMT; ++mi) v.nslot[mi] = max(v.nslot[mi], tk[mi].nrun);
  }
  return v;
}

template <typename SM>
__device__ __forceinline__ bool gl_wait(SM& sm, uint64_t* bar, uint32_t parity, int lane) {
  bool ok = true;
  if (lane == 0) {
    ok = !*reinterpret_cast<volatile int32_t*>(&sm.abort) && mbar_wait(bar, parity, kGlWaitNs);
    if (!ok) {
      set_err(sm.t.err_flag, LORA_ERR_TIMEOUT);
      atomicExch(&sm.abort, 1);
    }
  }
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int R>
__global__ void __launch_bounds__(kGlThreads, 1) gemm_lora_kernel(const __grid_constant__ GlParams p) {
  using Cfg = GlCfg<R>;
  using SM = GlSmem<R>;
  constexpr int RP = Cfg::RP;
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << kGlCM) - 1u);  // every CTA of the cluster
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  auto& sm = *reinterpret_cast<SM*>(smem_raw);
  const GlTail& q = sm.t;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  {
    static_assert(sizeof(GlTail) % 4 == 0, "tail size");
    const uint32_t* src = reinterpret_cast<const uint32_t*>(&p.t);
    uint32_t* dst = reinterpret_cast<uint32_t*>(&sm.t);
    for (int i = tid; i < static_cast<int>(sizeof(GlTail) / 4); i += kGlThreads) dst[i] = src[i];
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&p.tmX);
    prefetch_tmap(&p.tmXg);
    prefetch_tmap(&p.tmX2);
    prefetch_tmap(&p.tmW);
    prefetch_tmap(&p.tmW3);
    prefetch_tmap(&p.tmB);
    prefetch_tmap(&p.tmY);
  }
  if (tid == 0) {
    for (int s = 0; s < kGlStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kGlCM);  // every CTA of the cluster has consumed the slot
    }
    for (int b = 0; b < kGlBufs; ++b) {
      mbar_init(&sm.acc_full[b], 1);
      mbar_init(&sm.acc_empty[b], 4);
    }
    mbar_init(&sm.op_full, 4);
    mbar_init(&sm.op_empty, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (kGlCM > 1) {  // every CTA's barriers exist before a peer copies or commits into them
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  const uint32_t tmem = sm.tmem_base;
  pdl_launch_dependents();
  pdl_wait();  // v (and the segmentation) come from the launches before
  const bool aligned = (smem_u32(sm.st) & 1023u) == 0;
  if (!aligned && tid == 0) set_err(q.err_flag, LORA_ERR_UNSUPPORTED);

  const int crank = static_cast<int>(blockIdx.x) % kGlCM;
  const int u0 = static_cast<int>(blockIdx.x) / kGlCM, ustep = static_cast<int>(gridDim.x) / kGlCM;
  const int S = min(max(*q.num_segments, 0), q.max_segments);

  if (aligned && warp == 4) {
    // ============================== producer
    int slot = 0;
    uint32_t ph = 0, filled = 0, fill_par = 0;
    int cur_m = -1, cur_l = 0;
    GlView v{};
    GlTile t[kGlMT];
    int rr[kGlMT][4];
    auto advance = [&]() {
      filled |= 1u << slot;
      fill_par = (fill_par & ~(1u << slot)) | (ph << slot);
      if (++slot == kGlStages) {
        slot = 0;
        ph ^= 1u;
      }
    };
    bool ok = true;
    for (int u = u0; u < q.units && ok; u += ustep) {
      const GlUnit un = gl_unit(q, u, crank);
      if (un.mt != cur_m || un.ntl != cur_l) {
        v = gl_view(q, S, u, crank, lane, t);
        cur_m = un.mt;
        cur_l = un.ntl;
#pragma unroll
        for (int mi = 0; mi < kGlMT; ++mi) {
          if (t[mi].tlen > 0 && t[mi].row < 0) {
            // four rows per lane for the gathers; rows past the tile or with a
            // corrupt permutation entry read a valid row (never stored)
            int first = q.perm[t[mi].t0];
            if (first < 0 || first >= q.n_tokens) first = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = 4 * lane + j;
              const int r = i < t[mi].tlen ? q.perm[t[mi].t0 + i] : first;
              rr[mi][j] = (r >= 0 && r < q.n_tokens) ? r : first;
            }
          }
        }
      }
      if (!v.all) continue;  // the empty half of the last pairs: no work in any role of the cluster
      uint32_t xbytes = 0;
#pragma unroll
      for (int mi = 0; mi < kGlMT; ++mi) xbytes += t[mi].tlen > 0 ? Cfg::kX : 0;
      const int c0 = un.nt * kGlBN;
      // both tiles' rows as one box: two contiguous tiles, the second right after the first
      const bool xpair = LSG_GL_WIDE && kGlMT == 2 && t[0].tlen > 0 && t[0].row >= 0 &&
                         t[kGlMT - 1].tlen > 0 && t[kGlMT - 1].row == t[0].row + 128;
      for (int kb = 0; kb < q.k_blocks && ok; ++kb) {
        ok = gl_wait(sm, &sm.empty[slot], ph ^ 1u, lane);
        if (!ok) break;
        uint8_t* st = sm.st[slot];
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.full[slot], xbytes + static_cast<uint32_t>(Cfg::kW));
          if (xpair) {
            tma_load_2d(st, &p.tmX2, kb * 64, t[0].row, &sm.full[slot]);
          } else {
#pragma unroll
            for (int mi = 0; mi < kGlMT; ++mi)
              if (t[mi].tlen > 0 && t[mi].row >= 0)
                tma_load_2d(st + mi * Cfg::kX, &p.tmX, kb * 64, t[mi].row, &sm.full[slot]);
          }
          if constexpr (kGlCM > 1) {
            // this CTA's share of the W tile, into every CTA of the cluster
#pragma unroll
            for (int h = crank * (4 / kGlCM); h < (crank + 1) * (4 / kGlCM); ++h)
              tma_load_2d_mc(st + kGlMT * Cfg::kX + h * 8192, &p.tmW, c0 + h * 64, kb * 64, &sm.full[slot], kMask);
          } else if (q.w3d) {
            tma_load_3d(st + kGlMT * Cfg::kX, &p.tmW3, 0, kb * 64, c0 / 64, &sm.full[slot]);
          } else {
#pragma unroll
            for (int h = 0; h < 4; ++h)
              tma_load_2d(st + kGlMT * Cfg::kX + h * 8192, &p.tmW, c0 + h * 64, kb * 64, &sm.full[slot]);
          }
        }
        __syncwarp();  // the stage's byte count is registered before the gathers land
#pragma unroll
        for (int mi = 0; mi < kGlMT; ++mi)
          if (t[mi].tlen > 0 && t[mi].row < 0)
            tma_gather4(st + mi * Cfg::kX + lane * 512, &p.tmXg, kb * 64, rr[mi][0], rr[mi][1], rr[mi][2],
                        rr[mi][3], &sm.full[slot]);
        __syncwarp();
        advance();
      }
#pragma unroll
      for (int mi = 0; mi < kGlMT; ++mi) {
#pragma unroll
        for (int j = 0; j < kGlMaxRuns; ++j) {
          if (j >= v.nslot[mi] || !ok) break;
          ok = gl_wait(sm, &sm.empty[slot], ph ^ 1u, lane);
          if (!ok) break;
          uint8_t* st = sm.st[slot] + kGlMT * Cfg::kX;
          if (lane == 0) {
            if (j < t[mi].nrun) {
              mbar_arrive_expect_tx(&sm.full[slot], static_cast<uint32_t>(Cfg::kB));
#pragma unroll
              for (int h = 0; h < 4; ++h)
                tma_load_3d(st + h * RP * 128, &p.tmB, c0 + h * 64, 0, t[mi].a[j], &sm.full[slot]);
            } else {
              mbar_arrive(&sm.full[slot]);  // an empty slot: keeps the cluster's rings in step
            }
          }
          __syncwarp();
          advance();
        }
      }
    }
    if (!ok && lane == 0) {
      // no copy issued here may still be landing when the CTA leaves
      for (int s2 = 0; s2 < kGlStages; ++s2)
        if (filled & (1u << s2)) (void)mbar_wait(&sm.full[s2], (fill_par >> s2) & 1u, kGlWaitNs);
    }
  } else if (aligned && warp == 5) {
    // ============================== MMA issuer
    constexpr uint32_t kId = umma_idesc_bf16(128, kGlBN, 0, 1);
    int slot = 0, ui = 0, nop = 0, cur_m = -1, cur_l = 0;
    uint32_t ph = 0;
    GlView v{};
    GlTile t[kGlMT];
    bool ok = true;
    // a consumed slot goes back to the producers of every CTA of the cluster
    auto release = [&](int sl) {
      if constexpr (kGlCM > 1) umma_commit_mc(&sm.empty[sl], kMask);
      else umma_commit(&sm.empty[sl]);
    };
    for (int u = u0; u < q.units && ok; u += ustep) {
      const GlUnit un = gl_unit(q, u, crank);
      if (un.mt != cur_m || un.ntl != cur_l) {
        v = gl_view(q, S, u, crank, lane, t);
        cur_m = un.mt;
        cur_l = un.ntl;
      }
      if (!v.all) continue;
      const bool mine = v.own;  // no rows here: the cluster's slots are consumed, no MMAs
      const int buf = ui % kGlBufs;
      const uint32_t use = static_cast<uint32_t>(ui / kGlBufs);
      if (mine) {
        ok = gl_wait(sm, &sm.acc_empty[buf], (use & 1u) ^ 1u, lane);
        if (!ok) break;
        tc_fence_after();
      }
      for (int kb = 0; kb < q.k_blocks && ok; ++kb) {
        ok = gl_wait(sm, &sm.full[slot], ph, lane);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t xs = smem_u32(sm.st[slot]), ws = xs + kGlMT * Cfg::kX;
#pragma unroll
          for (int mi = 0; mi < kGlMT; ++mi) {
            if (t[mi].tlen <= 0) continue;
            const uint32_t acc = tmem + static_cast<uint32_t>((buf + mi) * kGlBN);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // x: K-major, 128 B swizzle; W: MN-major, 128 B swizzle, 64-column atoms 8 KB apart
              const uint64_t ad = umma_desc(xs + mi * Cfg::kX + k * 32, 16, 1024, 2);
              const uint64_t bd = umma_desc(ws + k * 16 * 128, 8192, 1024, 2);
              umma_bf16(acc, ad, bd, kId, kb > 0 || k > 0);
            }
          }
          release(slot);
        }
        __syncwarp();
        if (++slot == kGlStages) {
          slot = 0;
          ph ^= 1u;
        }
      }
#pragma unroll
      for (int mi = 0; mi < kGlMT; ++mi) {
        const uint32_t acc = tmem + static_cast<uint32_t>((buf + mi) * kGlBN);
#pragma unroll
        for (int j = 0; j < kGlMaxRuns; ++j) {
          if (j >= v.nslot[mi] || !ok) break;
          const bool run = j < t[mi].nrun;
          ok = (!run || gl_wait(sm, &sm.op_full, nop & 1, lane)) && gl_wait(sm, &sm.full[slot], ph, lane);
          if (!ok) break;
          tc_fence_after();
          if (lane == 0 && run) {
            const uint32_t bs = smem_u32(sm.st[slot]) + kGlMT * Cfg::kX;
#pragma unroll
            for (int k = 0; k < RP / 16; ++k) {
              const uint64_t bd = umma_desc(bs + k * 16 * 128, RP * 128, 1024, 2);
#pragma unroll
              for (int hl = 0; hl < 2; ++hl) {
                const uint64_t ad =
                    umma_desc(smem_u32(sm.opst + hl * Cfg::kVop) + k * 32, 16, 8 * RP * 2, umma_layout(RP * 2));
                umma_bf16(acc, ad, bd, kId, true);
              }
            }
            umma_commit(&sm.op_empty);
          }
          if (lane == 0) release(slot);
          __syncwarp();
          if (run) ++nop;
          if (++slot == kGlStages) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) break;
      if (mine) {
        if (lane == 0 && !(gl_withhold(4) && ui == 0)) umma_commit(&sm.acc_full[buf]);
        __syncwarp();
        ++ui;
      }
    }
    // every MMA issued here has completed before TMEM is released
    if (lane == 0) {
      umma_commit(&sm.drain);
      (void)mbar_wait(&sm.drain, 0, kGlWaitNs);
    }
    __syncwarp();
  } else if (aligned && warp < 4) {
    // ============================== epilogue: thread = tile row m
    const int m = warp * 32 + lane;
    const uint32_t tq = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int ui = 0, nop = 0, cur_m = -1, cur_l = 0, op_m = -1, op_j = -1, nstg = 0;
    bool any = false;
    GlTile t[kGlMT];
    int yrow[kGlMT];
    bool bad[kGlMT];
    bool ok = true;
    const float s = q.scale;
    for (int u = u0; u < q.units && ok; u += ustep) {
      const GlUnit un = gl_unit(q, u, crank);
      if (un.mt != cur_m || un.ntl != cur_l) {
        any = gl_tiles(q, S, un, lane, t);
        cur_m = un.mt;
        cur_l = un.ntl;
#pragma unroll
        for (int mi = 0; mi < kGlMT; ++mi) {
          yrow[mi] = -1;
          bad[mi] = false;
          if (m < t[mi].tlen) {
            yrow[mi] = t[mi].row >= 0 ? t[mi].row + m : q.perm[t[mi].t0 + m];
            if (yrow[mi] < 0 || yrow[mi] >= q.n_tokens) {
              bad[mi] = true;
              yrow[mi] = -1;
            }
          }
        }
      }
      if (!any) continue;
      if (un.nt == 0) {  // a corrupt permutation entry is flagged once per tile
#pragma unroll
        for (int mi = 0; mi < kGlMT; ++mi)
          if (bad[mi]) set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
      }
      const int buf = ui % kGlBufs;
      const uint32_t use = static_cast<uint32_t>(ui / kGlBufs);
      // ---- operand (s * v, bf16 hi + lo, K-major, 2*RP-byte swizzle) of each long segment
#pragma unroll
      for (int mi = 0; mi < kGlMT; ++mi) {
#pragma unroll
        for (int j = 0; j < kGlMaxRuns; ++j) {
          if (j >= t[mi].nrun || !ok) break;
          const int tm = un.mt + mi;
          const bool build = op_m != tm || op_j != j;
          // this row's v (zero outside the segment), loaded before the wait
          // for the previous operand's MMAs so the loads overlap them
          float4 vv[R / 4];
          if (build) {
            const bool mine = yrow[mi] >= 0 && m >= t[mi].lo[j] && m < t[mi].hi[j];
            const float4* vr = reinterpret_cast<const float4*>(q.v + static_cast<int64_t>(mine ? yrow[mi] : 0) * R);
#pragma unroll
            for (int e = 0; e < R / 4; ++e) vv[e] = mine ? vr[e] : make_float4(0.f, 0.f, 0.f, 0.f);
            // the shrink's k-partial slices, summed in slice order
            for (int pp = 1; pp < q.vparts && mine; ++pp) {
              const float4* vp = vr + pp * (q.vslice / 4);
#pragma unroll
              for (int e = 0; e < R / 4; ++e) {
                const float4 u = vp[e];
                vv[e].x += u.x;
                vv[e].y += u.y;
                vv[e].z += u.z;
                vv[e].w += u.w;
              }
            }
          }
          if (nop > 0) {
            ok = gl_wait(sm, &sm.op_empty, (nop - 1) & 1, lane);
            if (!ok) break;
          }
          if (build) {
            const uint32_t hrow = smem_u32(sm.opst) + static_cast<uint32_t>(m) * (RP * 2);
            const uint32_t lrow = smem_u32(sm.opst + Cfg::kVop) + static_cast<uint32_t>(m) * (RP * 2);
#pragma unroll
            for (int c = 0; c < RP / 8; ++c) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = 0.f;
              if (c < R / 8) {
                const float4 v0 = vv[2 * c], v1 = vv[2 * c + 1];
                f[0] = s * v0.x;
                f[1] = s * v0.y;
                f[2] = s * v0.z;
                f[3] = s * v0.w;
                f[4] = s * v1.x;
                f[5] = s * v1.y;
                f[6] = s * v1.z;
                f[7] = s * v1.w;
              }
              uint32_t hw[4], lw[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
                const float2 hf = __bfloat1622float2(h);
                const __nv_bfloat162 l = __floats2bfloat162_rn(f[2 * e] - hf.x, f[2 * e + 1] - hf.y);
                hw[e] = *reinterpret_cast<const uint32_t*>(&h);
                lw[e] = *reinterpret_cast<const uint32_t*>(&l);
              }
              const uint32_t ha = swz<Cfg::kSwM>(hrow + c * 16), la = swz<Cfg::kSwM>(lrow + c * 16);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ha), "r"(hw[0]), "r"(hw[1]),
                           "r"(hw[2]), "r"(hw[3])
                           : "memory");
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(la), "r"(lw[0]), "r"(lw[1]),
                           "r"(lw[2]), "r"(lw[3])
                           : "memory");
            }
            fence_proxy_async_smem();  // read by the tensor cores
            op_m = tm;
            op_j = j;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.op_full);
          ++nop;
        }
      }
      if (!ok) break;
      // ---- y = bf16(acc), 64 columns at a time.  A warp whose 32 rows are
      // contiguous rows of the tile stages them in shared memory (128 B
      // swizzle) and stores one TMA box; other rows go out as 16-byte stores.
      ok = gl_wait(sm, &sm.acc_full[buf], use & 1u, lane);
      if (!ok) break;
      tc_fence_after();
      const int c0 = un.nt * kGlBN, nstg0 = nstg;
#pragma unroll
      for (int mi = 0; mi < kGlMT; ++mi) {
        if (t[mi].tlen <= 0) continue;  // the same for every lane
        const bool box = t[mi].row >= 0 && warp * 32 + 32 <= t[mi].tlen;  // the same for every lane
        uint16_t* yp = yrow[mi] >= 0 ? q.y + static_cast<int64_t>(yrow[mi]) * q.ldy : nullptr;
#pragma unroll 1
        for (int c = 0; c < kGlBN / 64; ++c) {
          const int col = c0 + c * 64;
          if (col >= q.h_out) break;  // the same for every lane
          uint32_t a0[32], a1[32];
          tmem_ld32(tq + static_cast<uint32_t>((buf + mi) * kGlBN + c * 64), a0);
          tmem_ld32(tq + static_cast<uint32_t>((buf + mi) * kGlBN + c * 64 + 32), a1);
          tmem_ld_wait();
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const __nv_bfloat162 o0 = __floats2bfloat162_rn(__uint_as_float(a0[2 * e]), __uint_as_float(a0[2 * e + 1]));
            const __nv_bfloat162 o1 = __floats2bfloat162_rn(__uint_as_float(a1[2 * e]), __uint_as_float(a1[2 * e + 1]));
            w[e] = *reinterpret_cast<const uint32_t*>(&o0);
            w[16 + e] = *reinterpret_cast<const uint32_t*>(&o1);
          }
          if (box) {
            uint8_t* sb = sm.opst + warp * 8192 + (nstg & 1) * 4096;
            if (lane == 0) bulk_wait_read1();  // the store that last read this buffer is done with it
            __syncwarp();
            const uint32_t rowa = smem_u32(sb) + static_cast<uint32_t>(lane) * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(swz<7>(rowa + i * 16)), "r"(w[4 * i]),
                           "r"(w[4 * i + 1]), "r"(w[4 * i + 2]), "r"(w[4 * i + 3])
                           : "memory");
            fence_proxy_async_smem();  // read by the tensor copy
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.tmY, col, t[mi].row + warp * 32, sb);
              bulk_commit();
            }
            ++nstg;
          } else if (yp != nullptr) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (col + i * 8 < q.h_out)
                *reinterpret_cast<uint4*>(yp + col + i * 8) =
                    make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
      if (lane == 0) bulk_wait_read0();  // the staging area holds the next unit's operand
      __syncwarp();
      if (nstg != nstg0) op_m = -1;  // the cached operand was overwritten
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
      ++ui;
    }
  }
  if (aligned && warp < 4 && lane == 0) bulk_wait0();  // y stores complete before the CTA leaves
  tc_fence_before();
  __syncthreads();
  if (kGlCM > 1) {  // no CTA leaves while a peer may still copy or commit into it
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

namespace {

template <int R>
lora_status launch_gemm_lora_r(GlParams& prm, const void* x, int64_t ldx, const void* W, const void* B_pool,
                               cudaStream_t stream) {
  GlTail& t = prm.t;
  lora_status s;
  const uint64_t n = static_cast<uint64_t>(t.n_tokens);
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(t.h_in), n};
    const uint64_t str[1] = {static_cast<uint64_t>(ldx) * 2};
    const uint32_t box[2] = {64, 128}, box_g[2] = {64, 1};
    if ((s = encode_tmap_bf16(&prm.tmX, x, 2, dims, str, box, 128)) != LORA_OK) return s;
    if ((s = encode_tmap_bf16(&prm.tmXg, x, 2, dims, str, box_g, 128)) != LORA_OK) return s;
    const uint32_t box2[2] = {64, 256};
    if ((s = encode_tmap_bf16(&prm.tmX2, x, 2, dims, str, box2, 128)) != LORA_OK) return s;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(t.h_out), static_cast<uint64_t>(t.h_in)};
    const uint64_t str[1] = {static_cast<uint64_t>(t.h_out) * 2};
    const uint32_t box[2] = {64, 64};
    if ((s = encode_tmap_bf16(&prm.tmW, W, 2, dims, str, box, 128)) != LORA_OK) return s;
  }
  // W viewed as [h_out / 64][h_in][64] (a 64-column block's rows h_out apart,
  // the blocks 128 bytes apart): a [4][64][64] box is one W tile in the
  // stage's layout.  Only when every block is whole, so no box reads past W.
  t.w3d = 0;
  if (LSG_GL_WIDE && t.h_out % 64 == 0) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(t.h_in), static_cast<uint64_t>(t.h_out / 64)};
    const uint64_t str[2] = {static_cast<uint64_t>(t.h_out) * 2, 128};
    const uint32_t box[3] = {64, 64, 4};
    t.w3d = encode_tmap_bf16(&prm.tmW3, W, 3, dims, str, box, 128) == LORA_OK ? 1 : 0;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(t.h_out), static_cast<uint64_t>(R),
                              static_cast<uint64_t>(t.n_adapters)};
    const uint64_t str[2] = {static_cast<uint64_t>(t.h_out) * 2, static_cast<uint64_t>(t.h_out) * R * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(GlCfg<R>::RP), 1};
    if ((s = encode_tmap_bf16(&prm.tmB, B_pool, 3, dims, str, box, 128)) != LORA_OK) return s;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(t.h_out), n};
    const uint64_t str[1] = {static_cast<uint64_t>(t.ldy) * 2};
    const uint32_t box[2] = {64, 32};
    if ((s = encode_tmap_bf16(&prm.tmY, t.y, 2, dims, str, box, 128)) != LORA_OK) return s;
  }
  auto kern = gemm_lora_kernel<R>;
  const size_t smem = sizeof(GlSmem<R>);
  static_assert(sizeof(GlSmem<R>) <= 227 * 1024, "shared memory of one CTA");
  static std::mutex mu;
  static int groups_cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  int clusters = 0;  // co-resident clusters of kGlCM CTAs (one CTA per SM)
  {
    std::lock_guard<std::mutex> lk(mu);
    clusters = groups_cache[dev & 63];
  }
  cudaLaunchAttribute at[2];
  auto cluster_attr = [&](cudaLaunchAttribute& a) {
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = kGlCM;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
  };
  if (clusters == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return LORA_ERR_CUDA;
    if (kGlCM > 1) {
      cudaLaunchConfig_t occ{};
      occ.gridDim = dim3(kGlCM * 64);
      occ.blockDim = dim3(kGlThreads);
      occ.dynamicSmemBytes = smem;
      cluster_attr(at[0]);
      occ.attrs = at;
      occ.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &occ) != cudaSuccess) return LORA_ERR_CUDA;
    } else if (cudaDeviceGetAttribute(&clusters, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return LORA_ERR_CUDA;
    }
    clusters = std::max(1, clusters);
    std::lock_guard<std::mutex> lk(mu);
    groups_cache[dev & 63] = clusters;
  }
  // Whole waves of groups run as pairs.  Groups left over run as pairs too
  // when they fill more than half a wave (one more wave of pairs is shorter
  // than two waves of single tiles), else as single tiles in one short wave.
  if (kGlMT == 2) {
    const int groups = ceil_div(ceil_div(t.m_tiles, 2), kGlCM) * t.n_tiles;
    int whole = (groups / clusters) * clusters;
    if (2 * (groups - whole) > clusters) whole = groups;
    t.pair_units = whole;
    t.units = whole + 2 * (groups - whole);
  } else {
    t.pair_units = 0;
    t.units = ceil_div(t.m_tiles, kGlCM) * t.n_tiles;
  }
  cudaLaunchConfig_t cfg{};
  int na = 0;
  cfg.gridDim = dim3(std::max(1, std::min(clusters, t.units)) * kGlCM);
  cfg.blockDim = dim3(kGlThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  if (kGlCM > 1) cluster_attr(at[na++]);
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, prm));
}

}  // namespace

lora_status launch_gemm_lora(const GemmLoraCall& c, cudaStream_t stream) {
  const int n = c.seg.n_tokens;
  // 1. v of the long segments (tensor-tile kernel, shrink mode), when the batch can have any
  SgmvCall sh{};
  sh.mode = kModeShrink;
  sh.proj[0] = ProjArgs{c.x, c.A_pool, nullptr, nullptr, c.ldx, 0, c.h_in, 0, 1.0f};
  sh.n_proj = 1;
  sh.r = c.r;
  sh.n_adapters = c.n_adapters;
  sh.seg = c.seg;
  sh.v_out = c.v;
  sh.err_flag = c.err_flag;
  int32_t vparts = 1;
  sh.v_parts_max = std::min(LSG_GL_SHRINK_PARTS, kGlVParts);
  sh.v_parts = &vparts;
  const bool runs = sgmv_tc_applicable(sh);
  if (runs) {
    const lora_status s = launch_sgmv_tc(sh, stream);
    if (s != LORA_OK) return s;
  }
  // 2. y = x . W + the long segments' delta
  GlParams prm{};
  GlTail& t = prm.t;
  t.perm = c.seg.perm;
  t.seg_offsets = c.seg.seg_offsets;
  t.seg_adapter = c.seg.seg_adapter;
  t.num_segments = c.seg.num_segments;
  t.v = c.v;
  t.y = c.y;
  t.ldy = c.ldy;
  t.err_flag = c.err_flag;
  t.n_tokens = n;
  t.max_segments = c.seg.max_segments;
  t.n_adapters = c.n_adapters;
  t.h_in = c.h_in;
  t.h_out = c.h_out;
  t.m_tiles = ceil_div(n, 128);
  t.n_tiles = ceil_div(c.h_out, kGlBN);
  t.k_blocks = ceil_div(c.h_in, 64);
  t.use_runs = runs ? 1 : 0;
  t.vparts = runs ? vparts : 1;
  t.vslice = static_cast<int64_t>(n) * c.r;
  t.scale = c.scale;
  lora_status s;
  switch (c.r) {
    case 8: s = launch_gemm_lora_r<8>(prm, c.x, c.ldx, c.W, c.B_pool, stream); break;
    case 16: s = launch_gemm_lora_r<16>(prm, c.x, c.ldx, c.W, c.B_pool, stream); break;
    case 32: s = launch_gemm_lora_r<32>(prm, c.x, c.ldx, c.W, c.B_pool, stream); break;
    case 64: s = launch_gemm_lora_r<64>(prm, c.x, c.ldx, c.W, c.B_pool, stream); break;
    default: return LORA_ERR_UNSUPPORTED;
  }
  if (s != LORA_OK) return s;
  // 3. the short segments' delta, in place (the long ones are done)
  SgmvCall f{};
  f.mode = kModeFused;
  f.proj[0] = ProjArgs{c.x, c.A_pool, c.B_pool, c.y, c.ldx, c.ldy, c.h_in, c.h_out, c.scale};
  f.n_proj = 1;
  f.r = c.r;
  f.n_adapters = c.n_adapters;
  f.seg = c.seg;
  f.err_flag = c.err_flag;
  f.long_done = runs ? 1 : 0;
  return launch_sgmv_cc(f, stream);
}

}  // namespace lsg
