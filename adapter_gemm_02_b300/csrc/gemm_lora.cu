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
// gemm_lora_kernel: one CTA per SM, persistent, in clusters of CM CTAs that
// take CM consecutive token tiles of the same column tile together: CTA k of
// a cluster loads its own x rows and the k-th part of the W tile, which it
// multicasts to every CTA of the cluster (each W tile is read from L2 once per
// cluster instead of once per CTA); a ring slot is refilled only after every
// CTA of the cluster has consumed it.  Six warps:
//   warps 0-3  epilogue (warp w: TMEM lane quarter w; thread = tile row): the
//              v operand of each long segment, then y from the accumulator
//   warp 4     producer: TMA x tiles [128][64] (2-D box, or four-row gathers
//              through the permutation), W tiles [64][256] (four [64][64]
//              boxes, MN-major, 128 B swizzle), B tiles [r][256]
//   warp 5     TMEM allocation; one thread issues the MMAs (M = 128, N = 256)
// The two 256-column accumulators alternate, so the epilogue of one tile
// overlaps the main loop of the next.  Units (group of CM token tiles, column
// tile), column tiles inner, are dealt round robin over the clusters, so the
// units in flight together cover a few token tiles and all of W: both stay in
// L2.  The long segments' expand slots of a unit are as many in every CTA of
// the cluster (the most any of its token tiles has; a CTA with fewer fills
// the rest with empty slots), so the rings stay in step.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace lsg {

constexpr int kGlThreads = 192;
constexpr int kGlStages = 4;
constexpr int kGlBN = 256;     // output columns per tile (MMA N)
constexpr int kGlMaxRuns = 3;  // long segments (>= 64 tokens) a 128-token window can overlap
// Build-time knobs, set by measurement: clusters of 4 that share W tiles by
// multicast halved the L2 reads but ran slower (132 SMs hold whole clusters,
// and the four rings wait for each other), so CTAs run alone (CM = 1); the
// producer prefetches the x and W boxes of the k-block LSG_GL_PREFETCH stages
// ahead into L2, so the ring's refills find them there.
#ifndef LSG_GL_CM
#define LSG_GL_CM 1
#endif
#ifndef LSG_GL_PREFETCH
#define LSG_GL_PREFETCH 0
#endif
constexpr int kGlCM = LSG_GL_CM;  // CTAs per cluster sharing the W tiles (1, 2 or 4)
constexpr int kGlPrefetch = LSG_GL_PREFETCH;
static_assert(kGlCM == 1 || kGlCM == 2 || kGlCM == 4, "cluster size");
constexpr uint64_t kGlWaitNs = LSG_WAIT_LIMIT_NS;

struct GlTail {
  const int32_t* perm;
  const int32_t* seg_offsets;
  const int32_t* seg_adapter;
  const int32_t* num_segments;
  const float* v;  // [n][r] fp32: rows of long-segment tokens
  uint16_t* y;
  int64_t ldy;
  int32_t* err_flag;
  int32_t n_tokens, max_segments, n_adapters, h_in, h_out;
  int32_t m_tiles, n_tiles, k_blocks;
  int32_t use_runs;  // long segments' expands are fused here (their v was computed)
  float scale;
};

struct GlParams {
  CUtensorMap tmX;   // x [n][h_in], box {64, 128}, 128 B swizzle
  CUtensorMap tmXg;  // x, box {64, 1} (four-row gathers)
  CUtensorMap tmW;   // W [h_in][h_out], box {64, 64}, 128 B swizzle
  CUtensorMap tmB;   // B pool [P][r][h_out], box {64, RP, 1} (rows past r read zeros), 128 B swizzle
  GlTail t;
};

template <int R>
struct GlCfg {
  static constexpr int RP = R < 16 ? 16 : R;  // MMA K of the expand (rank 8 padded with zero rows)
  static constexpr int kX = 16384;            // x tile [128][64]
  static constexpr int kW = 32768;            // W tile [64][256]
  static constexpr int kStage = kX + kW;
  static constexpr int kB = RP * 512;         // B tile [RP][256] (in the W part of a stage)
  static constexpr int kVop = 128 * RP * 2;   // one bf16 operand [128][RP]
  static constexpr uint32_t kSwM = (RP * 2) / 16 - 1;
  static_assert(kB <= kW, "B tile fits a stage");
};

template <int R>
struct GlSmem {
  alignas(1024) uint8_t st[kGlStages][GlCfg<R>::kStage];
  alignas(1024) uint8_t vop[2][GlCfg<R>::kVop];  // hi, lo
  alignas(16) GlTail t;
  alignas(8) uint64_t full[kGlStages];
  uint64_t empty[kGlStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
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
  if (t.tlen <= 0) {  // a cluster's token tile past the batch: no rows, no segments
    t.row = -1;
    t.nrun = 0;
    return;
  }
  const int f = q.perm[t.t0];
  bool c = f >= 0 && f + t.tlen <= n;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = 4 * lane + j;
    if (i < t.tlen) c &= q.perm[t.t0 + i] == f + i;
  }
  t.row = __all_sync(0xffffffffu, c) ? f : -1;
  t.nrun = 0;
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

template <int R, int CM>
__global__ void __launch_bounds__(kGlThreads, 1) gemm_lora_kernel(const __grid_constant__ GlParams p) {
  using Cfg = GlCfg<R>;
  using SM = GlSmem<R>;
  constexpr int RP = Cfg::RP;
  constexpr uint16_t kMask = static_cast<uint16_t>((1u << CM) - 1u);  // every CTA of the cluster
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
    prefetch_tmap(&p.tmW);
    prefetch_tmap(&p.tmB);
  }
  if (tid == 0) {
    for (int s = 0; s < kGlStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], CM);  // every CTA of the cluster has consumed the slot
    }
    for (int b = 0; b < 2; ++b) {
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
  if (CM > 1) {  // every CTA's barriers exist before a peer copies or commits into them
    cluster_arrive_relaxed();
    cluster_wait_acquire();
  }
  const uint32_t tmem = sm.tmem_base;
  pdl_launch_dependents();
  pdl_wait();  // v (and the segmentation) come from the launches before
  const bool aligned = (smem_u32(sm.st) & 1023u) == 0;
  if (!aligned && tid == 0) set_err(q.err_flag, LORA_ERR_UNSUPPORTED);

  // units (group of CM token tiles, column tile), column tiles inner, dealt
  // round robin over the clusters: the units in flight together cover a few
  // token tiles and all of W, which stay in L2 (a contiguous range per
  // cluster would put all of x and W in flight)
  const int crank = static_cast<int>(blockIdx.x) % CM;
  const int units = ((q.m_tiles + CM - 1) / CM) * q.n_tiles;
  const int u0 = static_cast<int>(blockIdx.x) / CM, ustep = static_cast<int>(gridDim.x) / CM;
  const int S = min(max(*q.num_segments, 0), q.max_segments);
  // expand slots of a unit: the most long segments any token tile of the group overlaps
  auto group_runs = [&](int g) {
    int mx = 0;
#pragma unroll
    for (int k = 0; k < CM; ++k) {
      GlTile tk;
      gl_tile(q, S, g * CM + k, lane, tk);
      mx = max(mx, tk.nrun);
    }
    return mx;
  };

  if (aligned && warp == 4) {
    // ============================== producer
    int slot = 0;
    uint32_t ph = 0, filled = 0, fill_par = 0;
    int cur_m = -1, nslots_x = 0;
    GlTile t{};
    int rr[4] = {0, 0, 0, 0};
    auto advance = [&]() {
      filled |= 1u << slot;
      fill_par = (fill_par & ~(1u << slot)) | (ph << slot);
      if (++slot == kGlStages) {
        slot = 0;
        ph ^= 1u;
      }
    };
    bool ok = true;
    for (int u = u0; u < units && ok; u += ustep) {
      const int g = u / q.n_tiles, nt = u - g * q.n_tiles;
      const int mt = g * CM + crank;
      if (mt != cur_m) {
        gl_tile(q, S, mt, lane, t);
        nslots_x = CM > 1 ? group_runs(g) : t.nrun;
        cur_m = mt;
        if (t.tlen > 0 && t.row < 0) {
          // four rows per lane for the gathers; rows past the tile or with a
          // corrupt permutation entry read a valid row (never stored)
          int first = q.perm[t.t0];
          if (first < 0 || first >= q.n_tokens) first = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = 4 * lane + j;
            const int r = i < t.tlen ? q.perm[t.t0 + i] : first;
            rr[j] = (r >= 0 && r < q.n_tokens) ? r : first;
          }
        }
      }
      const int c0 = nt * kGlBN;
      for (int kb = 0; kb < q.k_blocks && ok; ++kb) {
        ok = gl_wait(sm, &sm.empty[slot], ph ^ 1u, lane);
        if (!ok) break;
        uint8_t* st = sm.st[slot];
        if (kGlPrefetch > 0 && lane == 0 && kb + kGlPrefetch < q.k_blocks) {
          // the boxes this CTA will load kGlPrefetch stages later, into L2 now
          const int kp = kb + kGlPrefetch;
          if (t.tlen > 0 && t.row >= 0) tma_prefetch_2d(&p.tmX, kp * 64, t.row);
#pragma unroll
          for (int h = crank * (4 / CM); h < (crank + 1) * (4 / CM); ++h) tma_prefetch_2d(&p.tmW, c0 + h * 64, kp * 64);
        }
        if (lane == 0) {
          // own x rows (none past the batch) and the whole W tile (every CTA's part)
          mbar_arrive_expect_tx(&sm.full[slot], static_cast<uint32_t>((t.tlen > 0 ? Cfg::kX : 0) + Cfg::kW));
          if (t.tlen > 0 && t.row >= 0) tma_load_2d(st, &p.tmX, kb * 64, t.row, &sm.full[slot]);
#pragma unroll
          for (int h = crank * (4 / CM); h < (crank + 1) * (4 / CM); ++h) {
            if constexpr (CM > 1)
              tma_load_2d_mc(st + Cfg::kX + h * 8192, &p.tmW, c0 + h * 64, kb * 64, &sm.full[slot], kMask);
            else
              tma_load_2d(st + Cfg::kX + h * 8192, &p.tmW, c0 + h * 64, kb * 64, &sm.full[slot]);
          }
        }
        __syncwarp();  // the stage's byte count is registered before the gathers land
        if (t.tlen > 0 && t.row < 0)
          tma_gather4(st + lane * 512, &p.tmXg, kb * 64, rr[0], rr[1], rr[2], rr[3], &sm.full[slot]);
        __syncwarp();
        advance();
      }
#pragma unroll
      for (int j = 0; j < kGlMaxRuns; ++j) {
        if (j >= nslots_x || !ok) break;
        ok = gl_wait(sm, &sm.empty[slot], ph ^ 1u, lane);
        if (!ok) break;
        uint8_t* st = sm.st[slot];
        if (lane == 0) {
          if (j < t.nrun) {
            mbar_arrive_expect_tx(&sm.full[slot], static_cast<uint32_t>(Cfg::kB));
#pragma unroll
            for (int h = 0; h < 4; ++h)
              tma_load_3d(st + Cfg::kX + h * RP * 128, &p.tmB, c0 + h * 64, 0, t.a[j], &sm.full[slot]);
          } else {
            mbar_arrive(&sm.full[slot]);  // an empty slot: keeps the cluster's rings in step
          }
        }
        __syncwarp();
        advance();
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
    int slot = 0, ui = 0, nop = 0, cur_m = -1, nslots_x = 0;
    uint32_t ph = 0;
    GlTile t{};
    bool ok = true;
    // a consumed slot goes back to the producers of every CTA of the cluster
    auto release = [&](int sl) {
      if constexpr (CM > 1) umma_commit_mc(&sm.empty[sl], kMask);
      else umma_commit(&sm.empty[sl]);
    };
    for (int u = u0; u < units && ok; u += ustep) {
      const int g = u / q.n_tiles;
      const int mt = g * CM + crank;
      if (mt != cur_m) {
        gl_tile(q, S, mt, lane, t);
        nslots_x = CM > 1 ? group_runs(g) : t.nrun;
        cur_m = mt;
      }
      const bool mine = t.tlen > 0;  // a token tile past the batch: slots consumed, no MMAs
      const int buf = ui & 1;
      const uint32_t acc = tmem + static_cast<uint32_t>(buf * kGlBN);
      if (mine) {
        ok = gl_wait(sm, &sm.acc_empty[buf], ((ui >> 1) & 1) ^ 1u, lane);
        if (!ok) break;
        tc_fence_after();
      }
      for (int kb = 0; kb < q.k_blocks && ok; ++kb) {
        ok = gl_wait(sm, &sm.full[slot], ph, lane);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          if (mine) {
            const uint32_t xs = smem_u32(sm.st[slot]), ws = xs + Cfg::kX;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // x: K-major, 128 B swizzle; W: MN-major, 128 B swizzle, 64-column atoms 8 KB apart
              const uint64_t ad = umma_desc(xs + k * 32, 16, 1024, 2);
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
      for (int j = 0; j < kGlMaxRuns; ++j) {
        if (j >= nslots_x || !ok) break;
        const bool run = j < t.nrun;
        ok = (!run || gl_wait(sm, &sm.op_full, nop & 1, lane)) && gl_wait(sm, &sm.full[slot], ph, lane);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          if (run) {
            const uint32_t bs = smem_u32(sm.st[slot]) + Cfg::kX;
#pragma unroll
            for (int k = 0; k < RP / 16; ++k) {
              const uint64_t bd = umma_desc(bs + k * 16 * 128, RP * 128, 1024, 2);
#pragma unroll
              for (int hl = 0; hl < 2; ++hl) {
                const uint64_t ad =
                    umma_desc(smem_u32(sm.vop[hl]) + k * 32, 16, 8 * RP * 2, umma_layout(RP * 2));
                umma_bf16(acc, ad, bd, kId, true);
              }
            }
          }
          release(slot);
          if (run) umma_commit(&sm.op_empty);
        }
        __syncwarp();
        if (run) ++nop;
        if (++slot == kGlStages) {
          slot = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (mine) {
        if (lane == 0) umma_commit(&sm.acc_full[buf]);
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
    int ui = 0, nop = 0, cur_m = -1, op_m = -1, op_j = -1, yrow = -1;
    GlTile t{};
    bool ok = true;
    const float s = q.scale;
    for (int u = u0; u < units && ok; u += ustep) {
      const int g = u / q.n_tiles, nt = u - g * q.n_tiles;
      const int mt = g * CM + crank;
      if (mt != cur_m) {
        gl_tile(q, S, mt, lane, t);
        cur_m = mt;
        yrow = -1;
        if (m < t.tlen) {
          yrow = t.row >= 0 ? t.row + m : q.perm[t.t0 + m];
          if (yrow < 0 || yrow >= q.n_tokens) {
            if (nt == 0) set_err(q.err_flag, LORA_ERR_BAD_ADAPTER_ID);
            yrow = -1;
          }
        }
      }
      if (t.tlen <= 0) continue;  // a token tile past the batch: nothing to store
      const int buf = ui & 1;
      // ---- operand (s * v, bf16 hi + lo, K-major, 2*RP-byte swizzle) of each long segment
#pragma unroll
      for (int j = 0; j < kGlMaxRuns; ++j) {
        if (j >= t.nrun || !ok) break;
        if (nop > 0) {
          ok = gl_wait(sm, &sm.op_empty, (nop - 1) & 1, lane);
          if (!ok) break;
        }
        if (op_m != mt || op_j != j) {
          const bool mine = yrow >= 0 && m >= t.lo[j] && m < t.hi[j];
          const float* vr = q.v + static_cast<int64_t>(mine ? yrow : 0) * R;
          const uint32_t hrow = smem_u32(sm.vop[0]) + static_cast<uint32_t>(m) * (RP * 2);
          const uint32_t lrow = smem_u32(sm.vop[1]) + static_cast<uint32_t>(m) * (RP * 2);
#pragma unroll
          for (int c = 0; c < RP / 8; ++c) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 0.f;
            if (mine && c < R / 8) {
              const float4 v0 = reinterpret_cast<const float4*>(vr)[2 * c];
              const float4 v1 = reinterpret_cast<const float4*>(vr)[2 * c + 1];
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
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ha), "r"(hw[0]), "r"(hw[1]), "r"(hw[2]),
                         "r"(hw[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(la), "r"(lw[0]), "r"(lw[1]), "r"(lw[2]),
                         "r"(lw[3])
                         : "memory");
          }
          fence_proxy_async_smem();  // read by the tensor cores
          op_m = mt;
          op_j = j;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.op_full);
        ++nop;
      }
      if (!ok) break;
      // ---- y = bf16(acc), 32 columns at a time, 16-byte stores of this row
      ok = gl_wait(sm, &sm.acc_full[buf], (ui >> 1) & 1, lane);
      if (!ok) break;
      tc_fence_after();
      uint16_t* yp = yrow >= 0 ? q.y + static_cast<int64_t>(yrow) * q.ldy : nullptr;
      const int c0 = nt * kGlBN;
#pragma unroll 1
      for (int c = 0; c < kGlBN / 32; ++c) {
        const int col = c0 + c * 32;
        if (col >= q.h_out) break;  // the same for every lane
        uint32_t a32[32];
        tmem_ld32(tq + static_cast<uint32_t>(buf * kGlBN + c * 32), a32);
        tmem_ld_wait();
        if (yp != nullptr) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (col + i * 8 < q.h_out) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 o = __floats2bfloat162_rn(__uint_as_float(a32[i * 8 + 2 * e]),
                                                               __uint_as_float(a32[i * 8 + 2 * e + 1]));
                w[e] = *reinterpret_cast<const uint32_t*>(&o);
              }
              *reinterpret_cast<uint4*>(yp + col + i * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
      ++ui;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CM > 1) {  // no CTA leaves while a peer may still copy or commit into it
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
  const GlTail& t = prm.t;
  lora_status s;
  const uint64_t n = static_cast<uint64_t>(t.n_tokens);
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(t.h_in), n};
    const uint64_t str[1] = {static_cast<uint64_t>(ldx) * 2};
    const uint32_t box[2] = {64, 128}, box_g[2] = {64, 1};
    if ((s = encode_tmap_bf16(&prm.tmX, x, 2, dims, str, box, 128)) != LORA_OK) return s;
    if ((s = encode_tmap_bf16(&prm.tmXg, x, 2, dims, str, box_g, 128)) != LORA_OK) return s;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(t.h_out), static_cast<uint64_t>(t.h_in)};
    const uint64_t str[1] = {static_cast<uint64_t>(t.h_out) * 2};
    const uint32_t box[2] = {64, 64};
    if ((s = encode_tmap_bf16(&prm.tmW, W, 2, dims, str, box, 128)) != LORA_OK) return s;
  }
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(t.h_out), static_cast<uint64_t>(R),
                              static_cast<uint64_t>(t.n_adapters)};
    const uint64_t str[2] = {static_cast<uint64_t>(t.h_out) * 2, static_cast<uint64_t>(t.h_out) * R * 2};
    const uint32_t box[3] = {64, static_cast<uint32_t>(GlCfg<R>::RP), 1};
    if ((s = encode_tmap_bf16(&prm.tmB, B_pool, 3, dims, str, box, 128)) != LORA_OK) return s;
  }
  auto kern = gemm_lora_kernel<R, kGlCM>;
  const size_t smem = sizeof(GlSmem<R>);
  static std::mutex mu;
  static int groups_cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  int clusters = 0;
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
  const int units = ceil_div(t.m_tiles, kGlCM) * t.n_tiles;
  cudaLaunchConfig_t cfg{};
  int na = 0;
  cfg.gridDim = dim3(std::max(1, std::min(clusters, units)) * kGlCM);
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
