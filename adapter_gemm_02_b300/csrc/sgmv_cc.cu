// SGMV on CUDA cores for short segments (decode), the HBM-bound regime.
//
// Punica: Multi-Tenant LoRA Serving (research.elamur.ai summary), "Summary":
// the per-adapter low-rank additions of a mixed batch are computed together,
// requests of one adapter grouped into segments; "Key points": rank is far
// below the hidden size (16 vs 4096).  For a decode segment the work is a few
// rank-r dot products per token, so time goes to streaming the adapter's A
// and B slabs from HBM; this kernel is built to keep HBM busy:
//
//  * Work item = (token tile of <= T tokens of one segment, projection).  A
//    cluster of C CTAs takes one item: CTA `rank` streams rows
//    [rank*k_chunk, +k_chunk) of A (split-K of the shrink) and columns
//    [rank*n_chunk, +n_chunk) of B (split-N of the expand).
//  * Partial v = x.A of each CTA is summed across the cluster through
//    distributed shared memory (fixed order, so every CTA holds identical v);
//    v never leaves the chip in the fused mode.
//  * One producer warp issues bulk (TMA) copies of A rows, gathered x rows,
//    B row pieces and gathered y rows into a 4-stage shared-memory ring
//    (16 KiB stages, mbarrier transaction counts); it runs ahead across items
//    so the next item's A slab streams while the current item is expanded.
//  * Four consumer warps: shrink with 16-byte A loads and fp32 FMAs, warp
//    shuffle + shared-memory split-K reduction; expand with 16-byte B loads,
//    a k-split over lanes reduced by shuffles, fp32 accumulate, one
//    round-to-nearest-even bf16 store of y (16-byte stores).
//  * Persistent grid: as many clusters as are co-resident; cluster g takes
//    items g, g+G, ... in tile-major order (all projections of a tile in a
//    row), read from the device-side segmentation without a host round trip.
//
// Modes: shrink (v -> device memory), expand (v from device memory, no
// cluster), fused (v on chip).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace lsg {

constexpr int kCW = 4;                 // consumer warps
constexpr int kCThreads = kCW * 32;    // consumer threads
constexpr int kThreads = kCThreads + 32;
constexpr int kStages = 4;
constexpr int kStageBytes = 16384;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

enum : int { kStShrink = 1, kStExpand = 2, kStFirst = 4, kStLast = 8, kStEnd = 16 };

struct CCProj {
  const uint16_t* x;
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* y;
  int64_t ldx, ldy;
  int32_t h_in, h_out;
  int32_t k_chunk, n_chunk;  // rows of A / columns of B per rank (multiples of 8)
  float scale;
};

struct CCParams {
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
  int32_t csplit;  // C
};

template <int R, int T>
struct CCCfg {
  // rows (shrink) or columns (expand) per stage: A/B part + x/y part fit a stage
  static constexpr int W = ((kStageBytes / ((R + T) * 2)) / 8) * 8;
  static constexpr int kPartBytes = W * R * 2;
  static constexpr int G = R / 8;           // shrink: 16-byte k-groups per A row
  static constexpr int L = kCThreads / G;   // shrink: row lanes
  static constexpr int KQ = R / 4;          // expand: lanes sharing one output vector (4 k each)
  static_assert(W >= 8, "stage too small");
  static_assert(kPartBytes + T * W * 2 <= kStageBytes, "stage overflow");
};

template <int T>
struct StageHdr {
  int32_t kind;
  int32_t proj;
  int32_t tlen;
  int32_t len;  // rows (shrink) or columns (expand) in this stage
  int32_t off;  // first row / column
  int32_t tok[T];
};

template <int R, int T>
struct CCSmem {
  alignas(128) uint8_t ring[kStages][kStageBytes];
  StageHdr<T> hdr[kStages];
  alignas(8) uint64_t full[kStages];
  uint64_t empty[kStages];
  float red[kCW][T][R];
  alignas(16) float vpart[T][R];
  alignas(16) float vfull[T][R];
};

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ float bf16_at(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}

__device__ __forceinline__ void consumer_sync() { named_bar_sync(1, kCThreads); }

// Locate token tile `tile` (tiles of <= T tokens, segment by segment) with a
// forward-only cursor over the segments (tile indices a CTA visits only grow).
// Executed by a full warp; returns false when `tile` is past the last tile.
template <int T>
__device__ bool find_tile(int& seg_base, int& tiles_before, int tile, int S, const int32_t* offs, int n,
                          int lane, int& seg, int& t0, int& tlen) {
  while (seg_base < S) {
    const int s = seg_base + lane;
    int off = 0, len = 0;
    if (s < S) {
      off = offs[s];
      const int end = offs[s + 1];
      len = (off >= 0 && end <= n && end >= off) ? end - off : 0;
    }
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
      const int Ls = __ffs(m) - 1;
      const int excl = __shfl_sync(0xffffffffu, inc - tl, Ls);
      const int o = __shfl_sync(0xffffffffu, off, Ls);
      const int l = __shfl_sync(0xffffffffu, len, Ls);
      seg = seg_base + Ls;
      t0 = o + (tile - tiles_before - excl) * T;
      tlen = min(T, o + l - t0);
      return true;
    }
    tiles_before += total;
    seg_base += 32;
  }
  return false;
}

template <int R, int T, int MODE>
__global__ void __launch_bounds__(kThreads) sgmv_cc_kernel(const __grid_constant__ CCParams p) {
  using Cfg = CCCfg<R, T>;
  constexpr int W = Cfg::W;
  constexpr bool kHasShrink = (MODE & kModeShrink) != 0;
  constexpr bool kHasExpand = (MODE & kModeExpand) != 0;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  auto& sm = *reinterpret_cast<CCSmem<R, T>*>(smem_raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = p.csplit;
  const int rank = static_cast<int>(blockIdx.x) % C;
  const int group = static_cast<int>(blockIdx.x) / C;
  const int ngroups = static_cast<int>(gridDim.x) / C;
  const bool do_cluster = kHasShrink && C > 1;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // The next launch may begin its prologue; it waits for our completion before
  // touching memory.  We wait for the launch that wrote the segmentation (and
  // v in the expand mode) before reading anything.
  pdl_launch_dependents();
  pdl_wait();

  if (warp == kCW) {
    // ============================== producer warp
    int slot = 0;
    uint32_t phase = 0;
    bool any = false, failed = false;
    const int S = min(max(*p.num_segments, 0), p.max_segments);
    int seg_base = 0, tiles_before = 0;
    int last_tile = -1, a = -1, t0 = 0, tlen = 0, tok = -1, ntok = 0;
    bool tile_ok = false;

    auto acquire = [&]() -> bool {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&sm.empty[slot], phase ^ 1u, kWaitLimitNs);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && lane == 0) set_err(p.err_flag, LORA_ERR_TIMEOUT);
      return ok;
    };
    auto advance = [&]() {
      if (++slot == kStages) {
        slot = 0;
        phase ^= 1u;
      }
    };

    for (int item = group; !failed; item += ngroups) {
      const int tile = item / p.n_proj;
      const int pj = item - tile * p.n_proj;
      if (tile != last_tile) {
        int seg;
        if (!find_tile<T>(seg_base, tiles_before, tile, S, p.seg_offsets, p.n_tokens, lane, seg, t0, tlen)) break;
        last_tile = tile;
        a = __shfl_sync(0xffffffffu, lane == 0 ? p.seg_adapter[seg] : 0, 0);
        tok = -1;
        if (lane < tlen) {
          tok = p.perm[t0 + lane];
          if (tok < 0 || tok >= p.n_tokens) {
            set_err(p.err_flag, LORA_ERR_BAD_ADAPTER_ID);
            tok = -1;
          }
        }
        ntok = __popc(__ballot_sync(0xffffffffu, tok >= 0));
        tile_ok = (a >= 0 && a < p.n_adapters);
        if (!tile_ok && lane == 0) set_err(p.err_flag, LORA_ERR_BAD_ADAPTER_ID);
      }
      if (!tile_ok) continue;  // every CTA of the cluster skips it alike
      const CCProj& pr = p.proj[pj];

      if (kHasShrink) {
        if (do_cluster) {
          if (any) cluster_wait_acquire();  // peers finished reading the previous partial v
          cluster_arrive_relaxed();
        }
        const int k0 = rank * pr.k_chunk;
        const int klen = max(0, min(pr.h_in, k0 + pr.k_chunk) - k0);
        const int nst = max(1, (klen + W - 1) / W);
        const int per = ((klen + nst - 1) / nst + 7) & ~7;
        const uint16_t* Aslab = pr.A + static_cast<int64_t>(a) * pr.h_in * R;
        for (int st = 0; st < nst && !failed; ++st) {
          const int r0 = k0 + st * per;
          const int rl = max(0, min(per, k0 + klen - r0));
          if (!acquire()) {
            failed = true;
            break;
          }
          StageHdr<T>& h = sm.hdr[slot];
          if (lane < T) h.tok[lane] = tok;
          if (lane == 0) {
            h.kind = kStShrink | (st == 0 ? kStFirst : 0) | (st == nst - 1 ? kStLast : 0);
            h.proj = pj;
            h.tlen = tlen;
            h.len = rl;
            h.off = r0;
          }
          __syncwarp();
          const uint32_t bytes = static_cast<uint32_t>(rl) * 2u * (R + ntok);
          if (lane == 0) {
            if (bytes) mbar_arrive_expect_tx(&sm.full[slot], bytes);
            else mbar_arrive(&sm.full[slot]);
          }
          __syncwarp();
          if (rl > 0) {
            uint8_t* st_base = sm.ring[slot];
            if (lane == 0) bulk_g2s(st_base, Aslab + static_cast<int64_t>(r0) * R, rl * R * 2, &sm.full[slot]);
            if (tok >= 0)
              bulk_g2s(st_base + Cfg::kPartBytes + lane * W * 2, pr.x + static_cast<int64_t>(tok) * pr.ldx + r0,
                       rl * 2, &sm.full[slot]);
          }
          advance();
        }
      }
      if (kHasExpand && !failed) {
        const int c0 = rank * pr.n_chunk;
        const int clen = max(0, min(pr.h_out, c0 + pr.n_chunk) - c0);
        const int nst = (clen + W - 1) / W;
        const int per = nst ? ((clen + nst - 1) / nst + 7) & ~7 : 0;
        const uint16_t* Bslab = pr.B + static_cast<int64_t>(a) * R * pr.h_out;
        for (int st = 0; st < nst; ++st) {
          const int cc = c0 + st * per;
          const int cl = max(0, min(per, c0 + clen - cc));
          if (!acquire()) {
            failed = true;
            break;
          }
          StageHdr<T>& h = sm.hdr[slot];
          if (lane < T) h.tok[lane] = tok;
          if (lane == 0) {
            h.kind = kStExpand | (st == 0 ? kStFirst : 0) | (st == nst - 1 ? kStLast : 0);
            h.proj = pj;
            h.tlen = tlen;
            h.len = cl;
            h.off = cc;
          }
          __syncwarp();
          const uint32_t bytes = static_cast<uint32_t>(cl) * 2u * (R + ntok);
          if (lane == 0) {
            if (bytes) mbar_arrive_expect_tx(&sm.full[slot], bytes);
            else mbar_arrive(&sm.full[slot]);
          }
          __syncwarp();
          if (cl > 0) {
            uint8_t* st_base = sm.ring[slot];
            for (int k = lane; k < R; k += 32)
              bulk_g2s(st_base + k * W * 2, Bslab + static_cast<int64_t>(k) * pr.h_out + cc, cl * 2,
                       &sm.full[slot]);
            if (tok >= 0)
              bulk_g2s(st_base + Cfg::kPartBytes + lane * W * 2, pr.y + static_cast<int64_t>(tok) * pr.ldy + cc,
                       cl * 2, &sm.full[slot]);
          }
          advance();
        }
      }
      if (do_cluster && !failed) {
        cluster_wait_acquire();   // all shrink partials of this item are published
        cluster_arrive_relaxed(); // (ours: nothing to publish)
      }
      any = true;
    }
    if (!failed && acquire()) {
      if (lane == 0) {
        sm.hdr[slot].kind = kStEnd;
        mbar_arrive(&sm.full[slot]);
      }
    }
    if (do_cluster && any) cluster_wait_acquire();
    return;
  }

  // ============================== consumer warps
  const int ct = tid;  // 0 .. kCThreads-1
  int slot = 0;
  uint32_t phase = 0;
  bool any = false;
  float acc[T][8];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;

  for (;;) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&sm.full[slot], phase, kWaitLimitNs);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) set_err(p.err_flag, LORA_ERR_TIMEOUT);
      return;
    }
    const StageHdr<T>& h = sm.hdr[slot];
    const int kind = h.kind;
    if (kind & kStEnd) break;
    const int tlen = h.tlen, len = h.len, off = h.off, pj = h.proj;
    const uint8_t* st_base = sm.ring[slot];

    if (kind & kStShrink) {
      if (kind & kStFirst) {
#pragma unroll
        for (int t = 0; t < T; ++t)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;
      }
      const int g = ct % Cfg::G, l = ct / Cfg::G;
      const uint16_t* As = reinterpret_cast<const uint16_t*>(st_base);
      const uint16_t* Xs = reinterpret_cast<const uint16_t*>(st_base + Cfg::kPartBytes);
      for (int j = l; j < len; j += Cfg::L) {
        const uint4 av = *reinterpret_cast<const uint4*>(As + j * R + g * 8);
        float af[8];
        unpack8(av, af);
#pragma unroll
        for (int t = 0; t < T; ++t) {
          if (t < tlen) {
            const float xv = bf16_at(Xs + t * W + j);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[t][e] = fmaf(xv, af[e], acc[t][e]);
          }
        }
      }
      if (kind & kStLast) {
        // ---- reduce partial v over this CTA: lanes (same g), then warps
#pragma unroll
        for (int t = 0; t < T; ++t) {
          if (t < tlen) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float v = acc[t][e];
#pragma unroll
              for (int o = Cfg::G; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
              acc[t][e] = v;
            }
          }
        }
        if (lane < Cfg::G) {
#pragma unroll
          for (int t = 0; t < T; ++t)
            if (t < tlen)
#pragma unroll
              for (int e = 0; e < 8; ++e) sm.red[warp][t][lane * 8 + e] = acc[t][e];
        }
        if (do_cluster && any) cluster_wait_acquire();  // peers done reading our previous vpart
        consumer_sync();
        for (int idx = ct; idx < tlen * R; idx += kCThreads) {
          const int t = idx / R, k = idx % R;
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kCW; ++w) s += sm.red[w][t][k];
          sm.vpart[t][k] = s;
        }
        consumer_sync();
        if (do_cluster) {
          cluster_arrive_release();
          cluster_wait_acquire();
          const uint32_t base = smem_u32(&sm.vpart[0][0]);
          for (int idx = ct; idx < tlen * R; idx += kCThreads) {
            float s = 0.f;
            for (int q = 0; q < C; ++q) s += ld_dsmem_f32(mapa_shared(base + idx * 4, q));
            (&sm.vfull[0][0])[idx] = s;
          }
          consumer_sync();
          cluster_arrive_relaxed();
        } else {
          for (int idx = ct; idx < tlen * R; idx += kCThreads) (&sm.vfull[0][0])[idx] = (&sm.vpart[0][0])[idx];
          consumer_sync();
        }
        any = true;
        if (MODE == kModeShrink && rank == 0) {
          for (int idx = ct; idx < tlen * R; idx += kCThreads) {
            const int t = idx / R, k = idx % R;
            const int tk = h.tok[t];
            if (tk >= 0) p.v_out[static_cast<int64_t>(tk) * R + k] = sm.vfull[t][k];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);  // header and data of this slot no longer read
    } else {
      // ---- expand stage: y[tok, off .. off+len) += s * vfull[t] . B[:, off .. off+len)
      if (MODE == kModeExpand && (kind & kStFirst)) {
        consumer_sync();  // every warp is done with the previous item's v
        for (int idx = ct; idx < tlen * R; idx += kCThreads) {
          const int t = idx / R, k = idx % R;
          const int tk = h.tok[t];
          sm.vfull[t][k] = tk >= 0 ? p.v_in[static_cast<int64_t>(tk) * R + k] : 0.f;
        }
        consumer_sync();
      }
      const CCProj& pr = p.proj[pj];
      const uint16_t* Bs = reinterpret_cast<const uint16_t*>(st_base);
      const uint16_t* Ys = reinterpret_cast<const uint16_t*>(st_base + Cfg::kPartBytes);
      const int nv = len >> 3;
      const int units = nv * tlen * Cfg::KQ;
      for (int ub = warp * 32; ub < units; ub += kCThreads) {
        const int u = ub + lane;
        const bool act = u < units;
        const int kq = u % Cfg::KQ;
        const int rest = u / Cfg::KQ;
        const int cv = act ? rest % nv : 0;
        const int t = act ? rest / nv : 0;
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = 0.f;
        if (act) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int k = kq * 4 + kk;
            const uint4 bv = *reinterpret_cast<const uint4*>(Bs + k * W + cv * 8);
            float bf[8];
            unpack8(bv, bf);
            const float vv = sm.vfull[t][k];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = fmaf(vv, bf[e], o[e]);
          }
        }
#pragma unroll
        for (int s = 1; s < Cfg::KQ; s <<= 1)
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] += __shfl_xor_sync(0xffffffffu, o[e], s);
        if (act && kq == 0) {
          const int tk = h.tok[t];
          if (tk >= 0) {
            const uint4 yv = *reinterpret_cast<const uint4*>(Ys + t * W + cv * 8);
            float yf[8];
            unpack8(yv, yf);
            uint4 outv;
            __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&outv);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              ob[i] = __floats2bfloat162_rn(yf[2 * i] + pr.scale * o[2 * i], yf[2 * i + 1] + pr.scale * o[2 * i + 1]);
            *reinterpret_cast<uint4*>(pr.y + static_cast<int64_t>(tk) * pr.ldy + off + cv * 8) = outv;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (do_cluster && any) cluster_wait_acquire();
}

// ------------------------------------------------------------------ host side

namespace {

struct KernelInfo {
  int max_groups = 0;  // co-resident clusters (or CTA groups) on the device
};

template <int R, int T, int MODE>
lora_status launch_rtm(const CCParams& prm, int items_bound, cudaStream_t stream) {
  auto kern = sgmv_cc_kernel<R, T, MODE>;
  const size_t smem = sizeof(CCSmem<R, T>);
  const int C = prm.csplit;
  const bool cluster = (MODE & kModeShrink) && C > 1;

  static std::mutex mu;
  static KernelInfo info[64][17];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
  KernelInfo ki;
  {
    std::lock_guard<std::mutex> lk(mu);
    ki = info[dev & 63][C];
  }
  if (ki.max_groups == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return LORA_ERR_CUDA;
    if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return LORA_ERR_CUDA;
    if (cluster) {
      cudaLaunchConfig_t cfg{};
      cudaLaunchAttribute at[1];
      cfg.gridDim = dim3(C * 1024);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
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
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess)
        return LORA_ERR_CUDA;
      if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return LORA_ERR_CUDA;
      ki.max_groups = std::max(1, per_sm * nsm / C);
    }
    std::lock_guard<std::mutex> lk(mu);
    info[dev & 63][C] = ki;
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
lora_status dispatch_mode(Mode m, const CCParams& prm, int items_bound, cudaStream_t st) {
  switch (m) {
    case kModeShrink: return launch_rtm<R, T, kModeShrink>(prm, items_bound, st);
    case kModeExpand: return launch_rtm<R, T, kModeExpand>(prm, items_bound, st);
    default: return launch_rtm<R, T, kModeFused>(prm, items_bound, st);
  }
}

template <int T>
lora_status dispatch_r(int r, Mode m, const CCParams& prm, int items_bound, cudaStream_t st) {
  switch (r) {
    case 8: return dispatch_mode<8, T>(m, prm, items_bound, st);
    case 16: return dispatch_mode<16, T>(m, prm, items_bound, st);
    case 32: return dispatch_mode<32, T>(m, prm, items_bound, st);
    case 64: return dispatch_mode<64, T>(m, prm, items_bound, st);
    default: return LORA_ERR_UNSUPPORTED;
  }
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
  // ranks per item: about 512 rows/columns per CTA, at most 8 (portable cluster)
  const int C = std::clamp(ceil_div(hmax, 512), 1, 8);
  // tokens per tile: small tiles when segments are short on average
  const double avg = static_cast<double>(n) / std::max(1, std::min(n, call.n_adapters));
  const int T = avg <= 2.5 ? 2 : 8;

  CCParams prm{};
  for (int i = 0; i < call.n_proj; ++i) {
    const ProjArgs& a = call.proj[i];
    CCProj& q = prm.proj[i];
    q.x = a.x;
    q.A = a.A;
    q.B = a.B;
    q.y = a.y;
    q.ldx = a.ldx;
    q.ldy = a.ldy;
    q.h_in = a.h_in;
    q.h_out = a.h_out;
    q.k_chunk = round_up(ceil_div(a.h_in, C), 8);
    q.n_chunk = round_up(ceil_div(a.h_out, C), 8);
    q.scale = a.scale;
  }
  prm.perm = call.seg.perm;
  prm.seg_offsets = call.seg.seg_offsets;
  prm.seg_adapter = call.seg.seg_adapter;
  prm.num_segments = call.seg.num_segments;
  prm.v_out = call.v_out;
  prm.v_in = call.v_in;
  prm.err_flag = call.err_flag;
  prm.n_proj = call.n_proj;
  prm.n_tokens = n;
  prm.max_segments = S_max;
  prm.n_adapters = call.n_adapters;
  prm.csplit = C;

  // upper bound of the number of tiles: sum over segments of ceil(len/T)
  const int64_t tiles = std::min<int64_t>(n, (static_cast<int64_t>(n) + static_cast<int64_t>(S_max) * (T - 1)) / T);
  const int items_bound = static_cast<int>(std::min<int64_t>(tiles * call.n_proj, 1 << 30));
  if (T == 2) return dispatch_r<2>(call.r, call.mode, prm, items_bound, stream);
  return dispatch_r<8>(call.r, call.mode, prm, items_bound, stream);
}

}  // namespace lsg
